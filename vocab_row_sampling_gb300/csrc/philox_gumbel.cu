// philox_gumbel.cu -- the sampler's noise, materialised: Philox4x32-10 words
// and their fp32 Gumbel values for a block of (row, column) pairs.
#include "drs_device.cuh"
#include "drs_internal.h"

namespace drs {

__global__ void __launch_bounds__(256) philox_gumbel_kernel(PhiloxKey key, int64_t row0,
                                                            int64_t rows, int64_t vocab,
                                                            uint32_t* bits, float* gumbel) {
    const int64_t groups_per_row = (vocab + 3) / 4;
    const int64_t total = rows * groups_per_row;
    const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
         t += step) {
        const int64_t r = t / groups_per_row;
        const int64_t g = t - r * groups_per_row;
        const uint4 w = noise_words(key, static_cast<uint64_t>(row0 + r),
                                    static_cast<uint64_t>(g));
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int64_t c = 4 * g + q;
            if (c < vocab) {
                const uint32_t word = word_of(w, q);
                const int64_t idx = r * vocab + c;
                if (bits) bits[idx] = word;
                if (gumbel) gumbel[idx] = gumbel_of_bits(word);
            }
        }
    }
}

}  // namespace drs

extern "C" drs_status drs_philox_gumbel(uint64_t seed, int64_t row0, int64_t rows,
                                        int64_t vocab, uint32_t* out_bits,
                                        float* out_gumbel, void* stream) {
    if (rows < 0 || row0 < 0 || vocab < 1) return DRS_ERR_INVALID_ARG;
    if (rows == 0 || (!out_bits && !out_gumbel)) return DRS_OK;
    const int64_t groups = rows * ((vocab + 3) / 4);
    const int sms = drs::sm_count();
    if (sms <= 0) return DRS_ERR_CUDA;
    int64_t blocks = (groups + 255) / 256;
    const int64_t max_blocks = static_cast<int64_t>(sms) * 16;
    if (blocks > max_blocks) blocks = max_blocks;
    const drs::PhiloxKey key{static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)};
    drs::philox_gumbel_kernel<<<static_cast<unsigned>(blocks), 256, 0,
                                static_cast<cudaStream_t>(stream)>>>(
        key, row0, rows, vocab, out_bits, out_gumbel);
    return drs::cuda_status(cudaGetLastError());
}
