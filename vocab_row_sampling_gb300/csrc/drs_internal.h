// drs_internal.h -- host-side helpers shared by the libdrs translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "drs.h"

namespace drs {

// Device flag raised by a bounded device-side wait that ran out of time, on
// the current device (address of a __device__ int, looked up once per
// device).
int* device_error_flag();

// A fresh 32-bit launch generation; tags of exchange records carry it so
// that records left in a workspace by an earlier launch never match.
uint32_t next_generation();

// Streaming multiprocessors of the current device.
int sm_count();

// Map a CUDA error to a status.
inline drs_status cuda_status(cudaError_t e) {
    return e == cudaSuccess ? DRS_OK : DRS_ERR_CUDA;
}

inline bool aligned(const void* p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

constexpr size_t kWorkspaceAlign = 256;

// The exact top-k kernel (topk.cu): every converged row of the call, or
// only the rows of a device list (row_list[0] the count, the rows from
// row_list[64]) that an earlier kernel on the stream wrote. Temperatures and
// keep flags are indexed by global slot (row0 + row) / canvas_len.
size_t exact_topk_workspace_bytes(int32_t k);
int32_t exact_topk_max_k();
drs_status exact_topk(const float* logits, int64_t rows, int64_t vocab, int64_t row_stride,
                      int64_t row0, const float* temps, int64_t canvas_len, const uint8_t* keep,
                      const int32_t* row_list, int32_t k, int32_t* out_ids, float* out_logprobs,
                      void* workspace, cudaStream_t stream);

}  // namespace drs
