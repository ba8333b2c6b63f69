// gdn_selftest.cu -- a wait that runs out on purpose, to check failure detection.
//
// Every wait of the library's kernels on an mbarrier is bounded: after the
// error block's wait limit it records GDN_ERR_TIMEOUT and the kernel winds
// down instead of hanging.  This entry point exercises that path in its
// plainest form: one thread waits, through the same bounded wait the kernels
// use, on an mbarrier that nothing ever arrives on.  No copy, MMA or other
// asynchronous operation is outstanding, so when the limit passes the kernel
// simply returns; the context stays usable.
#include "gdn_tc_ptx.cuh"

namespace gdn {
namespace {

__global__ void stuck_wait_kernel(int* err) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        tc::mbar_init(b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) tc::mbar_wait(b, 0, err);   // phase 0 never completes
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" int gdn_selftest_stuck_wait(cudaStream_t stream) {
    int st = GDN_OK;
    int* err = current_error_word(&st);
    if (err == nullptr) return st;
    stuck_wait_kernel<<<1, 32, 0, stream>>>(err);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
