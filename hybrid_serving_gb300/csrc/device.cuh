// device.cuh -- small device helpers shared by the kernels.
#pragma once
#include <cuda_bf16.h>
#include <atomic>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.h"
#include "meta.h"

namespace hsd {

// One-time launch setup (function attributes such as the dynamic shared-memory limit) is per device: a
// launcher keeps a flag per device ordinal and fills the current device's slot on its first call there.
constexpr int kMaxDevices = 64;
inline int device_slot() {
  int d = -1;
  return (cudaGetDevice(&d) == cudaSuccess && d >= 0 && d < kMaxDevices) ? d : -1;
}

// Programmatic dependent launch: a kernel launched with launch_pdl may start while the kernel before it in
// the stream drains.  Such a kernel calls pdl_wait() before it touches global memory (it returns once every
// earlier kernel in the stream has completed and its writes are visible), then pdl_trigger(), which lets the
// next kernel start launching once all of this kernel's blocks have begun.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// First error wins; kernels skip the offending work instead of trapping.
__device__ __forceinline__ void set_status(int32_t* st, int32_t code) {
  if (st) atomicCAS(st, 0, code);
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Convert 16 bytes of T to floats (4 for fp32, 8 for bf16).
__device__ __forceinline__ void cvt16(const float4& raw, float* out, float) {
  out[0] = raw.x; out[1] = raw.y; out[2] = raw.z; out[3] = raw.w;
}
__device__ __forceinline__ void cvt16(const float4& raw, float* out, __nv_bfloat16) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(b[i]);
    out[2 * i] = f.x;
    out[2 * i + 1] = f.y;
  }
}

struct Meta {
  const int32_t* m;
  __device__ __forceinline__ int32_t h(int i) const { return m[i]; }
  __device__ __forceinline__ const int32_t* seg(int s) const { return m + m[hsm::H_OFF_SEG] + s * hsm::kSegWords; }
  __device__ __forceinline__ const int32_t* tok(int t) const { return m + m[hsm::H_OFF_TOK] + t * hsm::kTokWords; }
  __device__ __forceinline__ const int32_t* span(int s) const { return m + m[hsm::H_OFF_SPAN] + s * hsm::kSpanWords; }
  __device__ __forceinline__ const int32_t* tile(int t) const { return m + m[hsm::H_OFF_TILE] + t * hsm::kTileWords; }
  __device__ __forceinline__ const int32_t* tile_spans() const { return m + m[hsm::H_OFF_TILE_SPAN]; }
  __device__ __forceinline__ const int32_t* chunk(int c) const { return m + m[hsm::H_OFF_CHUNK] + c * hsm::kChunkWords; }
  __device__ __forceinline__ const int32_t* page_ref() const { return m + m[hsm::H_OFF_PAGE_REF]; }
  __device__ __forceinline__ const int32_t* readout() const { return m + m[hsm::H_OFF_READOUT]; }
  __device__ __forceinline__ const int32_t* level_off() const { return m + m[hsm::H_OFF_LEVEL]; }
  __device__ __forceinline__ const int32_t* level_seg() const { return m + m[hsm::H_OFF_LEVEL_SEG]; }
  __device__ __forceinline__ const int32_t* scan() const { return m + m[hsm::H_OFF_SCAN]; }
  __device__ __forceinline__ const int32_t* scan_level_off() const { return m + m[hsm::H_OFF_SCAN_LEVEL]; }
};

}  // namespace hsd

// Host: check a launch, record failures.
namespace hsd {
// Launch with programmatic stream serialization allowed (see pdl_wait); errors surface through
// cudaGetLastError as for a <<<>>> launch.
template <typename... KArgs, typename... Args>
inline void launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  (void)cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
}  // namespace hsd

#define HS_LAUNCH_CHECK(what)                                                          \
  do {                                                                                 \
    cudaError_t e__ = cudaGetLastError();                                              \
    if (e__ != cudaSuccess) return hs::fail(HS_ECUDA, "%s: %s", what, cudaGetErrorString(e__)); \
    hs::count_launch();                                                                \
  } while (0)
