// Self-test of the library's failure detection: a bounded pipeline wait that runs out.
//
// Every tensor-core kernel of the library waits on mbarriers only through mbar_wait, whose
// wait ends after a fixed number of SM cycles: the waiting thread then raises the CTA's
// abort flag and the timeout bit of the device status word, the other waiters leave when
// they see the flag, copies already in flight are allowed to land, tensor memory is freed
// and the kernel returns, so the context stays usable.  No valid input makes a wait of the
// product kernels run out.  This kernel rebuilds that situation on purpose with a barrier
// nothing ever arrives on, so that the whole exit path can be run and checked:
//   warp 0  issues a real 4 KB bulk copy into shared memory, then drains it (a wait that
//           ignores the abort flag, as the copy producers of the GEMM kernels drain theirs);
//   warp 1  allocates and, at the end, frees 32 columns of tensor memory;
//   warp 2  waits on the barrier nothing arrives on, with the caller's short limit;
//   warp 3  waits on another such barrier under the normal limit and leaves on the flag.
// steps_out[0] collects one bit per stage that completed: 1 the copy landed, 2 the short
// wait gave up, 4 the second waiter left on the abort flag, 8 the kernel reached its end
// with its tensor memory freed.
#include "tc_common.cuh"

namespace moe {
namespace tc {

__global__ void __launch_bounds__(128, 1)
bounded_wait_selftest_kernel(const uint4* __restrict__ src, long long limit, int* __restrict__ status,
                             int32_t* __restrict__ steps_out) {
  __shared__ __align__(128) uint8_t buf[4096];
  __shared__ __align__(8) uint64_t bars[3];  // never, landed, never_either
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_word, steps;
  volatile int* abort_flag = &abort_word;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t never = smem_u32(&bars[0]), landed = smem_u32(&bars[1]), never_either = smem_u32(&bars[2]);
  if (threadIdx.x == 0) {
    mbar_init(never, 1);
    mbar_init(landed, 1);
    mbar_init(never_either, 1);
    abort_word = 0;
    steps = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_holder)),
                 "r"(32));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  grid_dep_wait();
  grid_dep_launch();
  if (warp == 0 && lane == 0) {
    mbar_expect_tx(landed, 4096);
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 4096, [%2];" ::"r"(
            smem_u32(buf)),
        "l"(src), "r"(landed)
        : "memory");
    if (mbar_wait(landed, 0, abort_flag, status, false)) atomicOr(&steps, 1);
  } else if (warp == 2 && lane == 0) {
    if (!mbar_wait_limit(never, 0, abort_flag, status, true, limit)) atomicOr(&steps, 2);
  } else if (warp == 3 && lane == 0) {
    if (!mbar_wait(never_either, 0, abort_flag, status, true) && *abort_flag) atomicOr(&steps, 4);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(32));
  }
  __syncthreads();
  if (threadIdx.x == 0) steps_out[0] = steps | 8;
}

}  // namespace tc
}  // namespace moe

extern "C" moe_status_t moe_selftest_bounded_wait(const void* src, long long limit_cycles, int32_t* steps_out,
                                                  moe_stream_t stream) {
  using namespace moe;
  if (!src || !steps_out || !aligned16(src)) return MOE_ERR_INVALID_ARG;
  if (limit_cycles < 1000 || limit_cycles > tc::WAIT_LIMIT_CYCLES) return MOE_ERR_INVALID_ARG;
  int* status = device_status_word();
  if (!status) return MOE_ERR_CUDA;
  return launch_kernel(tc::bounded_wait_selftest_kernel, dim3(1), dim3(128), 0, as_cuda(stream),
                       static_cast<const uint4*>(src), limit_cycles, status, steps_out);
}
