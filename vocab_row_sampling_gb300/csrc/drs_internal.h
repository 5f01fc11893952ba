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

// The current device's second stream and its fork and join events (created on
// first use): a call that runs part of its work beside the caller's stream
// records `fork` on it, makes the second stream wait for `fork`, and makes the
// caller's stream wait for `join` recorded after the second part.
bool side_stream(cudaStream_t* stream, cudaEvent_t* fork, cudaEvent_t* join);

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
// A row map for the exact top-k (the stash): the listed rows are entries e
// of a list, read from logits row row[e] with temperature temp[e]; outputs,
// and (when out_m is not null) the entry's max scaled logit and log of the
// sum of e^(s - max), are written at e.
struct ExactTopkMap {
    const int32_t* row;
    const float* temp;
    float* out_m;
    float* out_logs;
};
drs_status exact_topk(const float* logits, int64_t rows, int64_t vocab, int64_t row_stride,
                      int64_t row0, const float* temps, int64_t canvas_len, const uint8_t* keep,
                      const int32_t* row_list, int32_t k, int32_t* out_ids, float* out_logprobs,
                      void* workspace, cudaStream_t stream, const ExactTopkMap* map = nullptr);

// One call of the row statistics path: stats (argmax, sample, entropy and
// optionally probs) of every row, and with k > 0 the top-k logprobs of the
// converged rows (every row when keep is null). Temperatures and keep flags
// are indexed by global slot (row0 + row) / canvas_len.
struct RowCall {
    const float* logits;
    int64_t rows, vocab, row_stride;
    const float* temps;
    int64_t canvas_len;
    uint64_t seed;
    const uint64_t* seeds;  // null: one seed (`seed`); else n_seeds of them (HOST)
    int32_t n_seeds;
    int64_t row0;
    int64_t* argmax;
    int64_t* sample;
    float* entropy;
    drs_probs_dtype probs_dtype;
    void* probs;
    int64_t probs_row_stride;
    const uint8_t* keep;
    int32_t k;
    int32_t* out_ids;
    float* out_lp;
    bool stats;
    // Row map (the stash; all null otherwise): the call's rows are entries e
    // < *map_count (device) of a list, read from logits row map_row[e] with
    // temperature map_temp[e], every entry kept (keep and temps unused);
    // out_m / out_logs receive each entry's max scaled logit and log S.
    const int32_t* map_row;
    const float* map_temp;
    const int32_t* map_count;
    float* out_m;
    float* out_logs;
    // The caller has already written the row list, its header and every
    // listed entry's RowTemp (split_prep_targets): the call starts at pass 1
    // (the stash writes them with its own list).
    bool prepared;
};

// The fault-injection test hook (drs_test_inject_fault): the pending code,
// cleared by reading it.
int take_injected_fault();

// The test hook drs_test_two_pass: every row-statistics call takes the two
// passes, even where the one-read cluster kernel would.
bool two_pass_forced();

// Kernel timing (drs_kernel_timing): the ring slot of the calling row
// statistics call, or -1 when timing is off; the event to record before its
// kernel i (after the last kernel: i = kTimedKernels).
constexpr int kTimedKernels = 6;  // prep, pass 1, merge, pass 2, cluster, finish
constexpr int kTimedCalls = 64;
int kernel_timer_slot();
cudaEvent_t kernel_timer_event(int slot, int i);

// The two-pass row kernels (row_split.cu). The workspace starts with the
// hard-row list (count at [0], rows from [64]): rows whose top-k the exact
// kernel must finish. k is at most split_max_k().
size_t split_workspace_bytes(int64_t rows, int64_t vocab, int32_t k, int32_t n_seeds);
int32_t split_max_k();
int32_t split_max_seeds();
drs_status split_rows(const RowCall& c, void* workspace, cudaStream_t stream);

// Where a row call's workspace holds what its first kernel writes, for a
// caller that writes it itself (RowCall::prepared): the list header (word 0
// the hard-row count, 0 before pass 1; word 1 the list's length), the row
// list, and one RowTemp per listed entry (16 bytes: T, the quotient's 1/Te,
// y and mode).
struct SplitPrepTargets {
    int32_t* header;
    int32_t* list;
    void* row_temps;
};
SplitPrepTargets split_prep_targets(void* workspace, int64_t rows, int64_t vocab, int32_t k, int32_t n_seeds);

// How split_rows shares a call's rows on the current device: the first
// *head rows of its list go to the cluster kernel (*clusters clusters of
// *cluster_size CTAs resident at once), the others to the two passes on the
// *free_sms SMs the clusters leave. False when the call takes the two passes
// alone.
bool split_plan_query(int64_t rows, int64_t vocab, int32_t k, int32_t n_seeds, bool aligned16, int probs_dtype,
                      bool stats,
                      int64_t* head, int32_t* cluster_size, int32_t* clusters, int32_t* free_sms);

}  // namespace drs
