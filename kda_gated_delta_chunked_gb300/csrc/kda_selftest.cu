// kda_selftest.cu -- exercises the bounded-wait failure path of the kernels.
//
// The prefill kernels wait on mbarriers (TMA completion, tensor-core commits)
// with a time limit; when one runs out they record KDA_ERR_TIMEOUT in the
// workspace's device status word and return instead of hanging.  This entry
// point runs exactly that mechanism on an mbarrier nothing ever arrives on, so
// a test can check on a GPU that a wait which can never complete ends by
// itself and leaves the error where kda_get_device_status reads it.
#include "kda_common.cuh"
#include "kda_sm100.cuh"

namespace kda {

__global__ void kda_wait_that_runs_out(DeviceHeader* hdr, uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        sm100::mbar_init(&bar, 1);              // expects one arrival that never comes
        sm100::fence_mbar_init();
    }
    __syncthreads();
    const bool done = sm100::mbar_wait(&bar, 0, timeout_ns);
    if (threadIdx.x == 0) {
        hdr->total_chunks = 0;
        hdr->status = done ? KDA_OK : KDA_ERR_TIMEOUT;
    }
}

}  // namespace kda

extern "C" int kda_selftest_wait_timeout(const kda_desc* desc, int64_t timeout_ns, kda_stream_t stream) {
    if (!desc || !desc->workspace || desc->workspace_bytes < sizeof(kda::DeviceHeader)) return KDA_ERR_WORKSPACE;
    if (timeout_ns < 0 || timeout_ns > 1000000000LL) return KDA_ERR_INVALID_ARGUMENT;
    kda::kda_wait_that_runs_out<<<1, 32, 0, (cudaStream_t)stream>>>((kda::DeviceHeader*)desc->workspace,
                                                                      (uint64_t)timeout_ns);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
