// waitprobe.cu -- a check of the failure path of the bounded device waits.
//
// Every mbarrier wait of the tensor-core and bulk-copy kernels gives up after
// a time limit, raises GPT2_STATUS_TIMEOUT in the status word, tells the other
// roles of its CTA to leave (the abort flag), and the kernel returns instead of
// hanging.  This kernel runs that same wait (ptx::mbar_wait) on barriers that
// nothing ever completes, so the path can be exercised without a fault:
//   warp 0 waits with a short limit and gives up first;
//   warp 1 waits with the library's full limit (one second) and must leave as
//   soon as warp 0 has raised the abort flag.
// Both waits are bounded, so the kernel always ends; the context stays usable.
#include "common.cuh"
#include "ptx.cuh"

namespace gpt2k {

__global__ void __launch_bounds__(64) wait_probe_kernel(int* status, unsigned long long limit_ns) {
    using namespace ptx;
    __shared__ __align__(8) uint64_t never[2];
    __shared__ volatile int s_abort;
    if (threadIdx.x == 0) {
        s_abort = 0;
        mbar_init(smem_u32(&never[0]), 1);
        mbar_init(smem_u32(&never[1]), 1);
        fence_mbar_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0)
        (void)mbar_wait(smem_u32(&never[warp]), 0, &s_abort, status, warp == 0 ? limit_ns : WAIT_NS);
    __syncthreads();
}

int wait_probe(int* status, unsigned long long limit_ns, cudaStream_t st) {
    count_launch(), wait_probe_kernel<<<1, 64, 0, st>>>(status, limit_ns);
    GPT2_LAUNCH_CHECK();
    return GPT2_OK;
}

}  // namespace gpt2k
