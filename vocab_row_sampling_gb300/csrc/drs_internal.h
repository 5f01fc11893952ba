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

}  // namespace drs
