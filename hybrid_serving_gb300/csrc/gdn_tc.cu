// gdn_tc.cu -- Gated DeltaNet state pass on tcgen05 (bf16 inputs, d_k = d_v = 128).
//
// Flide, "Accelerating Decision Inference with Exact State Forking", section
// 3.2.2 (Eq. 4; children continue from the parent's end state by index),
// section 3.4 (checkpoint = saved end state of the first level), section 3.5
// (every node's chunks start at its first token).
//
// One CTA walks one node's chunks for one head, carrying the whole state S
// (d_v = 128 rows x d_k = 128) with d_v as the MMA M dimension.  For a chunk
// with inputs W, Ut, P, g (chunk-local pass) and Q, K (the stream):
//
//   D1 = S W^T            U  = Ut^T - D1         (U[j][t], j = row of S)
//   D2 = S Q^T            U' = U diag(e^{gC-g})
//   D3 = U P^T            O  = D2 diag(e^g) + D3   -> out[t][h][j]
//   D4 = U' K             S <- e^{gC} S + D4
//
// Warp 4 prefetches the next chunk (bulk copies of W, Ut, P, g from the
// workspace; TMA boxes of Q and K), warp 5 issues the MMAs from one thread,
// warps 0..3 (thread j = TMEM lane j = row j of S) keep S in fp32 registers,
// form U, O and the new S, and write the bf16 MMA operands (S, U, U') into
// shared memory.  Operands are bf16, accumulation fp32.  Every wait is
// bounded (HS_DEV_TIMEOUT).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "device.cuh"
#include "gdn_ws.h"
#include "tc_ptx.cuh"

using namespace hsm;
using hsd::Meta;

namespace {

constexpr int kD = 128;
constexpr int kThreads = 192;
constexpr long long kWaitCycles = 4000000000LL;
constexpr int HS_DEV_TIMEOUT = 4;
// shared memory (offsets from a 1024-aligned base)
constexpr int kOffS = 0;          // S  bf16 [128][128]: 2 slabs of [128][64]
constexpr int kOffU = 32768;      // U  bf16 [128][64]
constexpr int kOffUp = 49152;     // U' bf16 [128][64]
constexpr int kOffStage = 65536;  // 2 stages
constexpr int kStW = 0, kStQ = 16384, kStK = 32768, kStP = 49152, kStUt = 57344, kStG = 73728;
constexpr int kStageBytes = 74752;  // 73728 + 1024 (g padded)
constexpr int kSmem = kOffStage + 2 * kStageBytes;
constexpr uint32_t kStageTx = 16384 * 3 + 8192 + 16384 + 256;

constexpr uint32_t kIdesc64 = tc::idesc_bf16(128, 64, 0, 0);     // D[128x64], A, B K-major
constexpr uint32_t kIdesc128mn = tc::idesc_bf16(128, 128, 0, 1); // D[128x128], B N-major (K)

struct Prm {
  const int32_t* meta;
  int level, H, n_slots;
  const uint8_t* ws;
  float* state;
  __nv_bfloat16* out;
  int32_t* status;
};

__global__ void __launch_bounds__(kThreads, 1)
gdn_chain_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k, const Prm p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full[2], bar_empty[2], bar_s, bar_u, bar_d12, bar_d34, bar_done;
  __shared__ uint32_t tmem_slot;
  __shared__ float egs[2][64], dks[2][64], egc[2];
  __shared__ int abort_flag;
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);

  Meta M{p.meta};
  if (p.level >= M.h(H_N_LEVEL)) return;
  const int lo = M.level_off()[p.level], hi = M.level_off()[p.level + 1];
  if ((int)blockIdx.x >= hi - lo) return;
  const int seg = M.level_seg()[lo + blockIdx.x];
  const int32_t* sg = M.seg(seg);
  const int h = blockIdx.y;
  const int init = sg[S_INIT_SLOT], endslot = sg[S_END_SLOT];
  if (init >= p.n_slots || endslot >= p.n_slots) {
    if (threadIdx.x == 0) hsd::set_status(p.status, HS_DEV_BAD_SLOT);
    return;
  }
  const int c_off = sg[S_CHUNK_OFF], n_c = sg[S_N_CHUNK];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&bar_full[s], 1);
      tc::mbar_init(&bar_empty[s], 1);
    }
    tc::mbar_init(&bar_s, 128);
    tc::mbar_init(&bar_u, 128);
    tc::mbar_init(&bar_d12, 1);
    tc::mbar_init(&bar_d34, 1);
    tc::mbar_init(&bar_done, 1);
    tc::fence_mbar_init();
  }
  if (warp == 5) {
    tc::tmem_alloc(&tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  // TMEM columns: D1 [0,64) D2 [64,128) D3 [128,192) D4 [256,384)
  auto fail = [&]() {
    hsd::set_status(p.status, HS_DEV_TIMEOUT);
    atomicExch(&abort_flag, 1);
  };

  if (warp == 4) {
    // ----------------------------------------------------------- producer
    if (lane == 0) {
      tc::prefetch_tmap(&tm_q);
      tc::prefetch_tmap(&tm_k);
      int issued = 0;
      for (int ci = 0; ci < n_c; ++ci) {
        const int st = ci & 1;
        if (ci >= 2 && !tc::mbar_wait(&bar_empty[st], ((ci >> 1) - 1) & 1, kWaitCycles)) {
          fail();
          break;
        }
        if (*(volatile int*)&abort_flag) break;
        const int32_t* ch = M.chunk(c_off + ci);
        const int row0 = ch[C_ROW0];
        const uint8_t* w = p.ws + ((size_t)(c_off + ci) * p.H + h) * gdnws::kBytes;
        uint8_t* sb = smem + kOffStage + st * kStageBytes;
        tc::mbar_expect_tx(&bar_full[st], kStageTx);
        tc::bulk_load(sb + kStW, w + gdnws::kW, 16384, &bar_full[st]);
        tc::bulk_load(sb + kStUt, w + gdnws::kU, 16384, &bar_full[st]);
        tc::bulk_load(sb + kStP, w + gdnws::kP, 8192, &bar_full[st]);
        tc::bulk_load(sb + kStG, w + gdnws::kG, 256, &bar_full[st]);
        for (int half = 0; half < 2; ++half) {
          tc::tma_load_3d(sb + kStQ + half * 8192, &tm_q, half * 64, h, row0, &bar_full[st]);
          tc::tma_load_3d(sb + kStK + half * 8192, &tm_k, half * 64, h, row0, &bar_full[st]);
        }
        ++issued;
      }
      for (int ci = issued >= 2 ? issued - 2 : 0; ci < issued; ++ci)
        tc::mbar_wait(&bar_full[ci & 1], (ci >> 1) & 1, kWaitCycles);
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t sS = tc::smem_u32(smem + kOffS);
      const uint32_t sU = tc::smem_u32(smem + kOffU);
      const uint32_t sUp = tc::smem_u32(smem + kOffUp);
      bool ok = true;
      for (int ci = 0; ci < n_c && ok; ++ci) {
        const int st = ci & 1;
        const uint32_t sb = tc::smem_u32(smem + kOffStage + st * kStageBytes);
        if (!tc::mbar_wait(&bar_s, ci & 1, kWaitCycles) || !tc::mbar_wait(&bar_full[st], (ci >> 1) & 1, kWaitCycles)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        if (*(volatile int*)&abort_flag) {
          ok = false;
          break;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // D1 = S W^T, D2 = S Q^T   (K = d_k, 16 per step)
          const uint64_t a = tc::sdesc_sw128(sS + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024);
          const uint64_t bw = tc::sdesc_sw128(sb + kStW + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024);
          const uint64_t bq = tc::sdesc_sw128(sb + kStQ + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024);
          tc::mma_bf16_ss(tmem + 0, a, bw, kIdesc64, k > 0 ? 1u : 0u);
          tc::mma_bf16_ss(tmem + 64, a, bq, kIdesc64, k > 0 ? 1u : 0u);
        }
        tc::mma_commit(&bar_d12);
        if (!tc::mbar_wait(&bar_u, ci & 1, kWaitCycles)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // D3 = U P^T, D4 = U' K   (K = tokens, 16 per step)
          const uint64_t au = tc::sdesc_sw128(sU + k * 32, 16, 1024);
          const uint64_t aup = tc::sdesc_sw128(sUp + k * 32, 16, 1024);
          const uint64_t bp = tc::sdesc_sw128(sb + kStP + k * 32, 16, 1024);
          const uint64_t bk = tc::sdesc_sw128(sb + kStK + k * 2048, 8192, 1024);
          tc::mma_bf16_ss(tmem + 128, au, bp, kIdesc64, k > 0 ? 1u : 0u);
          tc::mma_bf16_ss(tmem + 256, aup, bk, kIdesc128mn, k > 0 ? 1u : 0u);
        }
        tc::mma_commit(&bar_d34);
        tc::mma_commit(&bar_empty[st]);
      }
      if (!ok) fail();
      tc::mma_commit(&bar_done);
      tc::mbar_wait(&bar_done, 0, kWaitCycles);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------- rows of the state
    const int j = threadIdx.x;  // row of S == TMEM lane
    const uint32_t lb = (uint32_t)(warp * 32) << 16;
    float S[kD];
    if (init >= 0) {
      const float4* src = reinterpret_cast<const float4*>(p.state + (((size_t)init * p.H + h) * kD + j) * kD);
#pragma unroll
      for (int i = 0; i < kD / 4; ++i) {
        const float4 v = src[i];
        S[4 * i] = v.x;
        S[4 * i + 1] = v.y;
        S[4 * i + 2] = v.z;
        S[4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < kD; ++i) S[i] = 0.f;
    }
    auto write_S = [&]() {  // bf16 row j of the A operand, 128-byte swizzle
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        uint4 v;
        v.x = tc::pack_bf16x2(S[c * 8 + 0], S[c * 8 + 1]);
        v.y = tc::pack_bf16x2(S[c * 8 + 2], S[c * 8 + 3]);
        v.z = tc::pack_bf16x2(S[c * 8 + 4], S[c * 8 + 5]);
        v.w = tc::pack_bf16x2(S[c * 8 + 6], S[c * 8 + 7]);
        *reinterpret_cast<uint4*>(smem + kOffS + gdnws::sw128_off(j, c * 8, 128)) = v;
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      tc::mbar_arrive(&bar_s);
    };
    write_S();
    bool ok = true;
    for (int ci = 0; ci < n_c; ++ci) {
      const int st = ci & 1, par = ci & 1;
      const uint8_t* sb = smem + kOffStage + st * kStageBytes;
      if (!__all_sync(~0u, tc::mbar_wait(&bar_full[st], (ci >> 1) & 1, kWaitCycles))) {
        ok = false;
        break;
      }
      const int32_t* ch = M.chunk(c_off + ci);
      const int row0 = ch[C_ROW0], len = ch[C_LEN];
      const float* g = reinterpret_cast<const float*>(sb + kStG);
      if (j < 64) {
        const float gC = g[len - 1];
        egs[par][j] = j < len ? expf(g[j]) : 0.f;
        dks[par][j] = j < len ? expf(gC - g[j]) : 0.f;
        if (j == 0) egc[par] = expf(gC);
      }
      tc::named_sync(1, 128);
      if (!__all_sync(~0u, tc::mbar_wait(&bar_d12, par, kWaitCycles))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      // U = Ut^T - D1,  U' = U diag(e^{gC-g})
      const __nv_bfloat16* ut = reinterpret_cast<const __nv_bfloat16*>(sb + kStUt);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t d1[32];
        tc::tmem_ld32(tmem + lb + half * 32, d1);
        tc::tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float u[8], up[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int t = half * 32 + c * 8 + e;
            u[e] = __bfloat162float(ut[t * kD + j]) - __uint_as_float(d1[c * 8 + e]);
            up[e] = u[e] * dks[par][t];
          }
          const int off = gdnws::sw128_off(j, half * 32 + c * 8, 128);
          uint4 a, b;
          a.x = tc::pack_bf16x2(u[0], u[1]);
          a.y = tc::pack_bf16x2(u[2], u[3]);
          a.z = tc::pack_bf16x2(u[4], u[5]);
          a.w = tc::pack_bf16x2(u[6], u[7]);
          b.x = tc::pack_bf16x2(up[0], up[1]);
          b.y = tc::pack_bf16x2(up[2], up[3]);
          b.z = tc::pack_bf16x2(up[4], up[5]);
          b.w = tc::pack_bf16x2(up[6], up[7]);
          *reinterpret_cast<uint4*>(smem + kOffU + off) = a;
          *reinterpret_cast<uint4*>(smem + kOffUp + off) = b;
        }
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      tc::mbar_arrive(&bar_u);
      if (!__all_sync(~0u, tc::mbar_wait(&bar_d34, par, kWaitCycles))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      // O = D2 diag(e^g) + D3  -> out[row0 + t][h][j]
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t d2[32], d3[32];
        tc::tmem_ld32(tmem + lb + 64 + half * 32, d2);
        tc::tmem_ld32(tmem + lb + 128 + half * 32, d3);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int t = half * 32 + e;
          if (t < len)
            p.out[((size_t)(row0 + t) * p.H + h) * kD + j] =
                __float2bfloat16_rn(fmaf(egs[par][t], __uint_as_float(d2[e]), __uint_as_float(d3[e])));
        }
      }
      // S <- e^{gC} S + D4
      const float ec = egc[par];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t d4[32];
        tc::tmem_ld32(tmem + lb + 256 + q * 32, d4);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) S[q * 32 + e] = fmaf(ec, S[q * 32 + e], __uint_as_float(d4[e]));
      }
      write_S();
    }
    if (!ok) {
      fail();
    } else if (endslot >= 0) {
      float4* dst = reinterpret_cast<float4*>(p.state + (((size_t)endslot * p.H + h) * kD + j) * kD);
#pragma unroll
      for (int i = 0; i < kD / 4; ++i) dst[i] = make_float4(S[4 * i], S[4 * i + 1], S[4 * i + 2], S[4 * i + 3]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 5) tc::tmem_dealloc(tmem, 512);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
  }
  return fn;
}

bool map_rows(CUtensorMap* m, const void* base, int H, long long T) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// State passes of every tree level on tensor cores, reading the compact
// workspace written by the chunk-local pass.
hs_status hs_gdn_chain_tc_launch(const hs_round_caps* caps, const int32_t* meta, int H, const void* q, const void* k,
                                 const uint8_t* ws, float* state, int n_slots, void* out, int32_t* status,
                                 cudaStream_t st) {
  CUtensorMap mq, mk;
  if (!map_rows(&mq, q, H, caps->max_tokens) || !map_rows(&mk, k, H, caps->max_tokens))
    return hs::fail(HS_ECUDA, "gdn: tensor map encoding failed");
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(gdn_chain_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem + 1024) !=
        cudaSuccess)
      return hs::fail(HS_ECUDA, "gdn_chain_tc: cannot raise the shared-memory limit");
    configured = true;
  }
  for (int lev = 0; lev < caps->max_levels && caps->max_segments > 0; ++lev) {
    Prm prm{meta, lev, H, n_slots, ws, state, (__nv_bfloat16*)out, status};
    gdn_chain_tc_kernel<<<dim3(caps->max_segments, H), kThreads, kSmem + 1024, st>>>(mq, mk, prm);
    HS_LAUNCH_CHECK("gdn_chain_tc");
  }
  return HS_OK;
}
