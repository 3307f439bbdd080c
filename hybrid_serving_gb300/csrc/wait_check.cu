// wait_check.cu -- the failure path of the bounded device waits, run on purpose.
//
// Every wait of the tcgen05 kernels on a shared-memory barrier gives up after
// a cycle limit: the kernel records HS_DEV_TIMEOUT in the caller's status
// word, lets the copies it has in flight land, frees its tensor memory and
// returns, so the context stays usable and the host learns of the failure
// from the status word.  One CTA here takes that path deterministically: it
// holds tensor memory and a bulk copy in flight while two of its warps wait,
// each with one of the two polling helpers the kernels use, on a barrier that
// nothing ever completes.
#include <cuda_runtime.h>

#include "device.cuh"
#include "tc_ptx.cuh"

namespace {

constexpr long long kDrainCycles = 4000000000LL;  // the copy in flight always lands: this never runs out
constexpr int kCopyBytes = 1024;
__device__ __align__(16) uint8_t g_copy_src[kCopyBytes];

__global__ void __launch_bounds__(64, 1) wait_timeout_kernel(long long wait_cycles, int32_t* status, long long* elapsed) {
  __shared__ __align__(1024) uint8_t buf[kCopyBytes];
  __shared__ uint64_t bar_copy, bar_never[2];
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar_copy, 1);
    tc::mbar_init(&bar_never[0], 1);  // nothing arrives on these
    tc::mbar_init(&bar_never[1], 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_slot, 32);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (threadIdx.x == 0) {  // a copy in flight while the waits run out
    tc::mbar_expect_tx(&bar_copy, kCopyBytes);
    tc::bulk_load(buf, g_copy_src, kCopyBytes, &bar_copy);
  }
  __syncwarp();
  // warp 0: the suspending poll (try_wait); warp 1: the spinning poll (test_wait); both voted as in the kernels
  const long long t0 = clock64();
  const bool ok = warp == 0 ? __all_sync(~0u, tc::mbar_wait(&bar_never[0], 0, wait_cycles))
                            : __all_sync(~0u, tc::mbar_wait_spin(&bar_never[1], 0, wait_cycles));
  const long long dt = clock64() - t0;
  if (!ok && lane == 0) hsd::set_status(status, HS_DEV_TIMEOUT);
  if (lane == 0 && elapsed) elapsed[warp] = dt;
  // the drain: the issuing thread waits for its copy before the block may exit
  if (threadIdx.x == 0 && !tc::mbar_wait(&bar_copy, 0, kDrainCycles)) hsd::set_status(status, HS_DEV_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem_slot, 32);
}

}  // namespace

extern "C" hs_status hs_debug_wait_timeout(int64_t wait_cycles, int32_t* dev_status, int64_t* dev_elapsed,
                                           void* stream) {
  HS_CHECK_ARG(dev_status, "null status word");
  HS_CHECK_ARG(wait_cycles >= 1 && wait_cycles <= (1LL << 31), "wait_cycles %lld outside [1, 2^31]",
               (long long)wait_cycles);
  wait_timeout_kernel<<<1, 64, 0, (cudaStream_t)stream>>>((long long)wait_cycles, dev_status,
                                                         reinterpret_cast<long long*>(dev_elapsed));
  HS_LAUNCH_CHECK("wait_timeout");
  return HS_OK;
}
