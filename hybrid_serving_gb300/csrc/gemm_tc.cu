// gemm_tc.cu -- batch-invariant bf16 GEMM on tcgen05 for sm_103a.
//
//   C[M, N] = A[M, K] . B[N, K]^T  (+ R[M, N])      bf16 in, fp32 accumulate, C and R bf16 or fp32
//
// Flide, "Accelerating Decision Inference with Exact State Forking",
// section 3.5: every matrix product sums each output element in a fixed
// order whatever the number of rows.  Here every output tile is 128 x 256,
// there is no split-K, and the K loop runs in the same 64-wide stages and
// 16-wide MMA steps for any M, so a row's result does not depend on which
// other rows share the launch.
//
// Persistent: one CTA per SM walks the output tiles t = blockIdx.x, + grid,
// ... in row-block-major order (the CTAs working at one time share their A
// rows, and B -- the weights -- stays in L2).  Warp 0 streams A and B tiles
// with TMA into a 4-stage ring (128-byte swizzle; rows of B past N read as
// zeros); warp 1 owns all 512 TMEM columns as two 256-column accumulators and
// issues tcgen05.mma (M=128, N=256, K=16) from one elected lane of the
// converged warp; warps 2..5 read an accumulator back (thread = row) 64 bytes
// of each row at a time, add the optional residual (TMA-loaded two pieces
// ahead into a shared staging buffer), write the piece into a second staging
// buffer and store it with one TMA store per 128 rows x 64 bytes (C in bf16
// rounded to nearest, or fp32: a residual stream kept in fp32), while the
// MMAs of the next tile fill the other accumulator.  Waits are bounded and
// report HS_DEV_TIMEOUT through the status word; the epilogue warps take
// every decision together, so a timeout never leaves one at a barrier.
//
// The SwiGLU variant (kGlu) takes B's rows in blocks of 128 gate rows followed
// by the 128 up rows of the same output columns, so a 256-wide tile holds both
// halves of 128 outputs: its epilogue writes silu(gate) * up, computed in fp32
// from the two accumulator halves and rounded to bf16 once.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "device.cuh"
#include "tc_ptx.cuh"

namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStages = 4;
constexpr int kStageA = BM * BK * 2;  // 16 KB
constexpr int kStageB = BN * BK * 2;  // 32 KB
constexpr int kRing = kStages * (kStageA + kStageB);  // 192 KB
constexpr int kStg = BM * 64;                          // a staging buffer: 128 rows x 64 bytes
constexpr int kSmem = kRing + 4 * kStg;                // + C and R pieces, two each: 224 KB
constexpr int kThreads = 192;
constexpr long long kWaitCycles = 4000000000LL;
constexpr uint32_t kIdesc = tc::idesc_bf16(BM, BN, 0, 0);

template <typename CT>
struct GemmParams {
  int M, N, K;
  CT* C;
  long long ldc;
  const CT* R;  // optional residual, same layout and type as C
  long long ldr;
  int32_t* status;
};

__device__ __forceinline__ float silu_f(float x) { return x / (1.f + expf(-x)); }

// 64 bytes of a row: 16 fp32 or 32 bf16 values
template <typename CT>
struct Piece;
template <>
struct Piece<float> {
  static constexpr int kCols = 16;
  static __device__ __forceinline__ void load(uint32_t taddr, uint32_t (&v)[32]) {
    tc::tmem_ld16(taddr, *reinterpret_cast<uint32_t(*)[16]>(v));
  }
  // v + residual (from shared memory) into 64 bytes of shared memory
  static __device__ __forceinline__ void put(const uint32_t (&v)[32], const uint8_t* res, uint8_t* dst) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float4 o = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]), __uint_as_float(v[4 * q + 2]),
                             __uint_as_float(v[4 * q + 3]));
      if (res) {
        const float4 r = tc::lds_f4(tc::smem_u32(res) + 16 * q);
        o.x += r.x; o.y += r.y; o.z += r.z; o.w += r.w;
      }
      tc::sts_f4(tc::smem_u32(dst) + 16 * q, o);
    }
  }
};
template <>
struct Piece<__nv_bfloat16> {
  static constexpr int kCols = 32;
  static __device__ __forceinline__ void load(uint32_t taddr, uint32_t (&v)[32]) { tc::tmem_ld32(taddr, v); }
  static __device__ __forceinline__ void put(const uint32_t (&v)[32], const uint8_t* res, uint8_t* dst) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float f[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(v[8 * q + i]);
      if (res) {
        float rr[8];
        const uint4 rw = tc::lds_u4(tc::smem_u32(res) + 16 * q);
        hsd::cvt16(*reinterpret_cast<const float4*>(&rw), rr, __nv_bfloat16());
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] += rr[i];
      }
      tc::sts_u4(tc::smem_u32(dst) + 16 * q, make_uint4(tc::pack_bf16x2(f[0], f[1]), tc::pack_bf16x2(f[2], f[3]),
                                                        tc::pack_bf16x2(f[4], f[5]), tc::pack_bf16x2(f[6], f[7])));
    }
  }
};

template <typename CT, bool kGlu>
__global__ void __launch_bounds__(kThreads, 1)
gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_r,
                    const GemmParams<CT> p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full[kStages], bar_empty[kStages], bar_acc[2], bar_free[2], bar_done, bar_r[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag, epi_go;
  // aligned up to 1024 bytes by pointer arithmetic on the shared array, so every access through smem stays
  // a shared-memory access (an integer round trip would turn them into generic loads and stores)
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nk = p.K / BK;
  const int n_tn = (p.N + BN - 1) / BN, n_tiles = ((p.M + BM - 1) / BM) * n_tn;
  // this CTA's tiles: blockIdx.x, + gridDim.x, ... (row block t / n_tn, column block t % n_tn)
  const int n_mine = (int)blockIdx.x < n_tiles ? (n_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&bar_full[s], 1);
      tc::mbar_init(&bar_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bar_acc[b], 1);     // accumulator b complete (MMA commit)
      tc::mbar_init(&bar_free[b], 128);  // accumulator b read out (every epilogue thread)
    }
    tc::mbar_init(&bar_done, 1);
    tc::mbar_init(&bar_r[0], 1);  // residual pieces landed
    tc::mbar_init(&bar_r[1], 1);
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      tc::prefetch_tmap(&tm_a);
      tc::prefetch_tmap(&tm_b);
      int issued = 0;  // stages over all tiles
      bool ok = true;
      for (int j = 0; j < n_mine && ok; ++j) {
        const int t = (int)blockIdx.x + j * (int)gridDim.x;
        const int m0 = (t / n_tn) * BM, n0 = (t % n_tn) * BN;
        for (int kb = 0; kb < nk; ++kb, ++issued) {
          const int s = issued % kStages;
          if (issued >= kStages && !tc::mbar_wait(&bar_empty[s], ((issued / kStages) - 1) & 1, kWaitCycles)) {
            hsd::set_status(p.status, HS_DEV_TIMEOUT);
            atomicExch(&abort_flag, 1);
            ok = false;
            break;
          }
          if (*(volatile int*)&abort_flag) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * (kStageA + kStageB);
          uint8_t* sb = sa + kStageA;
          tc::mbar_expect_tx(&bar_full[s], kStageA + kStageB);
          tc::tma_load_2d(sa, &tm_a, kb * BK, m0, &bar_full[s]);
          tc::tma_load_2d(sb, &tm_b, kb * BK, n0, &bar_full[s]);
        }
      }
      // drain: the last copies have landed before the CTA leaves
      for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
        tc::mbar_wait(&bar_full[i % kStages], (i / kStages) & 1, kWaitCycles);
    }
  } else if (warp == 1) {
    // converged warp: voted waits, one elected lane issues; a K step adds a constant to the descriptors
    bool ok = true;
    int used = 0;  // stages consumed over all tiles
    for (int j = 0; j < n_mine && ok; ++j) {
      const int b = j & 1;
      // accumulator b is free once the epilogue has read tile j - 2 out of it
      if (j >= 2 && !__all_sync(~0u, tc::mbar_wait(&bar_free[b], ((j - 2) >> 1) & 1, kWaitCycles))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint32_t acc = tmem + 256 * b;
      for (int kb = 0; kb < nk; ++kb, ++used) {
        const int s = used % kStages;
        if (!__all_sync(~0u, tc::mbar_wait(&bar_full[s], (used / kStages) & 1, kWaitCycles))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t sa = tc::smem_u32(smem + s * (kStageA + kStageB));
        const uint64_t da = tc::sdesc_sw128(sa, 16, 1024), db = tc::sdesc_sw128(sa + kStageA, 16, 1024);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          const uint64_t off = (uint64_t)((k * 32) >> 4);
          tc::mma_bf16_ss_w(acc, da + off, db + off, kIdesc, (kb > 0 || k > 0) ? 1u : 0u);
        }
        tc::mma_commit_w(&bar_empty[s]);
        if (*(volatile int*)&abort_flag) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
      tc::mma_commit_w(&bar_acc[b]);
    }
    if (!ok && lane == 0) {
      hsd::set_status(p.status, HS_DEV_TIMEOUT);
      atomicExch(&abort_flag, 1);
    }
    // every MMA issued has completed before the CTA leaves and TMEM is freed
    tc::mma_commit_w(&bar_done);
    __all_sync(~0u, tc::mbar_wait(&bar_done, 0, kWaitCycles));
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5, barrier 1)
    using PC = Piece<CT>;
    static_assert(!kGlu || sizeof(CT) == 2, "the SwiGLU epilogue writes bf16");
    constexpr int kOutCols = kGlu ? BN / 2 : BN;          // output columns per tile
    constexpr int kPieces = kOutCols / PC::kCols;          // per tile (even)
    const int quarter = warp % 4;            // TMEM lanes this warp may read
    const int r = quarter * 32 + lane;
    const bool issuer = r == 0;
    const uint32_t lanes = (uint32_t)(quarter * 32) << 16;
    uint8_t* cst = smem + kRing;            // C pieces: cst + b * kStg
    uint8_t* rst = smem + kRing + 2 * kStg;  // R pieces
    const bool has_r = p.R != nullptr;
    // the residual piece g (over all tiles) of this CTA: TMA into rst[g & 1]
    auto load_r = [&](int g) {
      const int j = g / kPieces, c = g % kPieces;
      if (!has_r || j >= n_mine) return;
      const int t = (int)blockIdx.x + j * (int)gridDim.x;
      tc::mbar_expect_tx(&bar_r[g & 1], kStg);
      tc::tma_load_2d(rst + (g & 1) * kStg, &tm_r, (t % n_tn) * kOutCols + c * PC::kCols, (t / n_tn) * BM,
                      &bar_r[g & 1]);
    };
    if (issuer) {
      tc::prefetch_tmap(&tm_c);
      if (has_r) tc::prefetch_tmap(&tm_r);
      load_r(0);
      load_r(1);
    }
    int stored = 0;  // pieces over all tiles
    for (int j = 0; j < n_mine; ++j) {
      // one decision for the four warps: go on unless a role gave up
      if (issuer) epi_go = !*(volatile int*)&abort_flag;
      tc::named_sync(1, 128);
      if (!epi_go) break;
      const int b = j & 1;
      const int t = (int)blockIdx.x + j * (int)gridDim.x;
      const int m0 = (t / n_tn) * BM, n0 = (t % n_tn) * kOutCols;  // (n0: the tile's first output column)
      if (!__all_sync(~0u, tc::mbar_wait(&bar_acc[b], (j >> 1) & 1, kWaitCycles))) {  // warp-wide: ld is collective
        hsd::set_status(p.status, HS_DEV_TIMEOUT);
        atomicExch(&abort_flag, 1);  // (this tile goes on with whatever it holds; the next one stops)
      }
      tc::fence_after_sync();
#pragma unroll 1
      for (int c = 0; c < kPieces; ++c, ++stored) {
        const int pb = stored & 1;
        uint32_t v[32], vu[32];
        PC::load(tmem + lanes + 256 * b + c * PC::kCols, v);
        if constexpr (kGlu) tc::tmem_ld32(tmem + lanes + 256 * b + BN / 2 + c * PC::kCols, vu);  // the up half
        tc::tmem_wait_ld();
        if (c == kPieces - 1) {  // the accumulator is read out: the MMAs of tile j + 2 may start
          tc::fence_before_sync();
          tc::mbar_arrive(&bar_free[b]);
        }
        if (has_r && !__all_sync(~0u, tc::mbar_wait(&bar_r[pb], (stored >> 1) & 1, kWaitCycles))) {
          hsd::set_status(p.status, HS_DEV_TIMEOUT);
          atomicExch(&abort_flag, 1);
        }
        if (issuer && stored >= 2) tc::bulk_wait_read_but1();  // the store of piece stored - 2 has read cst[pb]
        tc::named_sync(1, 128);
        if constexpr (kGlu) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(silu_f(__uint_as_float(v[i])) * __uint_as_float(vu[i]));
        }
        PC::put(v, has_r ? rst + pb * kStg + r * 64 : nullptr, cst + pb * kStg + r * 64);
        tc::fence_proxy_async_smem();
        tc::named_sync(1, 128);
        if (issuer) {
          if (n0 + c * PC::kCols < (kGlu ? p.N / 2 : p.N)) {  // (a piece wholly past the output is not stored)
            tc::tma_store_2d(&tm_c, n0 + c * PC::kCols, m0, cst + pb * kStg);
            tc::bulk_commit();
          }
          load_r(stored + 2);  // rst[pb] is read by every row (barrier above)
        }
      }
    }
    if (issuer) {
      tc::bulk_wait_all();  // the stores have completed
      // residual pieces loaded ahead but not used (the loop stopped early) land before the CTA leaves
      if (has_r) {
        const int n_loaded = min(stored + 2, n_mine * kPieces);
        for (int g = stored; g < n_loaded; ++g) tc::mbar_wait(&bar_r[g & 1], (g >> 1) & 1, kWaitCycles);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
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

bool map_2d(CUtensorMap* m, const void* base, long long rows, long long cols, long long ld, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {BK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// C or R [rows, cols] (leading dimension ld) in pieces of 128 rows x 64 bytes, unswizzled
bool map_piece(CUtensorMap* m, const void* base, long long rows, long long cols, long long ld, bool f32) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int es_b = f32 ? 4 : 2;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * es_b};
  cuuint32_t box[2] = {(cuuint32_t)(64 / es_b), (cuuint32_t)BM};
  cuuint32_t es[2] = {1, 1};
  return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
            dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace {

// the launch shared by both entry points: C[M, Nout] from A[M, K] and B[N, K] (Nout = N, or N / 2 with kGlu)
template <bool kGlu>
hs_status gemm_launch(int32_t M, int32_t N, int32_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                      void* C, int64_t ldc, const void* R, int64_t ldr, hs_dtype c_dtype, int32_t* dev_status,
                      void* stream) {
  const int n_out = kGlu ? N / 2 : N;
  HS_CHECK_ARG(lda >= K && ldb >= K && ldc >= n_out && (!R || ldr >= n_out), "leading dimensions too small");
  HS_CHECK_ARG(lda % 8 == 0 && ldb % 8 == 0 && ldc % 8 == 0 && (!R || ldr % 8 == 0),
               "leading dimensions must be multiples of 8 elements");
  HS_CHECK_ARG((((uintptr_t)A | (uintptr_t)B | (uintptr_t)C | (uintptr_t)R) & 15) == 0,
               "pointers must be 16-byte aligned");
  if (M == 0) return HS_OK;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return hs::fail(HS_ECUDA, "no CUDA device");
  CUtensorMap ma, mb;
  CUtensorMap mc, mr;
  const bool f32 = c_dtype == HS_F32;
  if (!map_2d(&ma, A, M, K, lda, BM) || !map_2d(&mb, B, N, K, ldb, BN) || !map_piece(&mc, C, M, n_out, ldc, f32) ||
      !map_piece(&mr, R ? R : C, M, n_out, R ? ldr : ldc, f32))
    return hs::fail(HS_ECUDA, "gemm: tensor map encoding failed");
  static std::atomic<bool> configured[hsd::kMaxDevices];  // zero-initialised: per device
  const int slot = hsd::device_slot();
  if (slot < 0) return hs::fail(HS_ECUDA, "gemm: no usable CUDA device");
  if (!configured[slot].load()) {
    if (cudaFuncSetAttribute(gemm_bf16_tc_kernel<__nv_bfloat16, kGlu>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmem + 1024) != cudaSuccess ||
        (!kGlu && cudaFuncSetAttribute(gemm_bf16_tc_kernel<float, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmem + 1024) != cudaSuccess))
      return hs::fail(HS_ECUDA, "gemm: cannot raise the shared-memory limit");
    configured[slot].store(true);
  }
  static std::atomic<int> sm_count[hsd::kMaxDevices];  // per device, 0 until read
  int n_sm = sm_count[slot].load();
  if (n_sm <= 0) {
    if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, slot) != cudaSuccess || n_sm <= 0)
      return hs::fail(HS_ECUDA, "gemm: cannot read the SM count");
    sm_count[slot].store(n_sm);
  }
  const long long n_tiles = (long long)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const dim3 grid((unsigned)(n_tiles < n_sm ? n_tiles : n_sm));  // persistent: one CTA per SM
  if (!kGlu && c_dtype == HS_F32) {
    GemmParams<float> prm{M, N, K, (float*)C, ldc, (const float*)R, ldr, dev_status};
    gemm_bf16_tc_kernel<float, false><<<grid, kThreads, kSmem + 1024, (cudaStream_t)stream>>>(ma, mb, mc, mr, prm);
  } else {
    GemmParams<__nv_bfloat16> prm{M, N, K, (__nv_bfloat16*)C, ldc, (const __nv_bfloat16*)R, ldr, dev_status};
    gemm_bf16_tc_kernel<__nv_bfloat16, kGlu><<<grid, kThreads, kSmem + 1024, (cudaStream_t)stream>>>(ma, mb, mc, mr,
                                                                                                    prm);
  }
  HS_LAUNCH_CHECK("gemm_bf16");
  return HS_OK;
}

}  // namespace

extern "C" hs_status hs_gemm_bf16(int32_t M, int32_t N, int32_t K, const void* A, int64_t lda, const void* B,
                                  int64_t ldb, void* C, int64_t ldc, const void* R, int64_t ldr, hs_dtype c_dtype,
                                  int32_t* dev_status, void* stream) {
  HS_CHECK_ARG(A && B && C, "null argument");
  if (c_dtype != HS_BF16 && c_dtype != HS_F32) return hs::fail(HS_EUNSUPPORTED, "gemm: C dtype %d", c_dtype);
  HS_CHECK_ARG(M >= 0 && N > 0 && K > 0, "bad shape %d x %d x %d", M, N, K);
  if (N % 128 != 0 || K % BK != 0)
    return hs::fail(HS_EUNSUPPORTED, "N (%d) must be a multiple of 128 and K (%d) of %d", N, K, BK);
  return gemm_launch<false>(M, N, K, A, lda, B, ldb, C, ldc, R, ldr, c_dtype, dev_status, stream);
}

extern "C" hs_status hs_gemm_bf16_swiglu(int32_t M, int32_t N2, int32_t K, const void* A, int64_t lda, const void* B,
                                         int64_t ldb, void* C, int64_t ldc, int32_t* dev_status, void* stream) {
  HS_CHECK_ARG(A && B && C, "null argument");
  HS_CHECK_ARG(M >= 0 && N2 > 0 && K > 0, "bad shape %d x %d x %d", M, N2, K);
  if (N2 % BN != 0 || K % BK != 0)
    return hs::fail(HS_EUNSUPPORTED, "N2 (%d) must be a multiple of %d and K (%d) of %d", N2, BN, K, BK);
  return gemm_launch<true>(M, N2, K, A, lda, B, ldb, C, ldc, nullptr, 0, HS_BF16, dev_status, stream);
}
