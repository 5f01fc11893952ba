// scale.cu -- the temperature-scaled logits, scaled = x / max(T, 1e-10),
// elementwise (page "vllm.model_executor.models.diffusion_gemma_sampler",
// sample_row_stats_reference: logits.float() / temp.clamp(min=1e-10)). The
// quotient is the routine the row kernels use (ScaledQuotient), with
// infinities kept, so this entry point exposes it to exhaustive checks.
#include "drs_device.cuh"
#include "drs_internal.h"

namespace drs {

__global__ void __launch_bounds__(256) scaled_logits_kernel(const float* __restrict__ x,
                                                            int64_t n, float temp,
                                                            float* __restrict__ out) {
    const ScaledQuotient sq = ScaledQuotient::of(fmaxf(temp, kTempFloor));
    const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += step)
        out[i] = sq.exact(x[i]);
}

}  // namespace drs

extern "C" drs_status drs_scaled_logits(const float* logits, int64_t n, float temp,
                                        float* out, void* stream) {
    if (n < 0) return DRS_ERR_INVALID_ARG;
    if (n == 0) return DRS_OK;
    if (!logits || !out || !drs::aligned(logits, 4) || !drs::aligned(out, 4))
        return DRS_ERR_INVALID_ARG;
    const int sms = drs::sm_count();
    if (sms <= 0) return DRS_ERR_CUDA;
    int64_t blocks = (n + 255) / 256;
    if (blocks > static_cast<int64_t>(sms) * 32) blocks = static_cast<int64_t>(sms) * 32;
    drs::scaled_logits_kernel<<<static_cast<unsigned>(blocks), 256, 0,
                                static_cast<cudaStream_t>(stream)>>>(logits, n, temp, out);
    return drs::cuda_status(cudaGetLastError());
}
