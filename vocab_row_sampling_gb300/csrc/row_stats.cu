// row_stats.cu -- the C entry points of the row statistics and the top-k
// logprobs (page "vllm.model_executor.models.diffusion_gemma_sampler":
// sample_row_stats, sample_row_stats_reference, stash_converged_logprobs,
// _lp_topk_kernel): argument checks, workspace layout, and the calls into the
// two-pass row kernels (row_split.cu) and the exact top-k kernel (topk.cu).
//
// drs_row_stats_topk: the row kernels give the statistics of every row and,
// for k <= 64, the top-k of every converged row whose candidates fit their
// lists; the exact kernel then finishes the rows listed as hard (no
// threshold, or too many candidates) on the same stream. For k > 64 the row
// statistics run alone and the exact kernel takes every converged row.
#include <atomic>
#include <climits>
#include <mutex>

#include "drs_device.cuh"
#include "drs_internal.h"

namespace drs {
namespace {

// The fault-injection hook (drs_test_inject_fault).
std::atomic<int> g_inject_fault{0};
// The two-pass hook (drs_test_two_pass).
std::atomic<int> g_two_pass{0};

drs_status check_stats_args(const float* logits, int64_t rows, int64_t vocab, int64_t row_stride,
                            const float* temps, int64_t canvas_len, int64_t row0, int64_t* argmax,
                            int64_t* sample, float* entropy, drs_probs_dtype probs_dtype,
                            void* probs, int64_t probs_row_stride) {
    if (rows < 0 || row0 < 0 || canvas_len < 1) return DRS_ERR_INVALID_ARG;
    if (vocab < 1 || row_stride < vocab) return DRS_ERR_INVALID_ARG;
    if (vocab > DRS_MAX_VOCAB) return DRS_ERR_UNSUPPORTED;
    if (!logits || !temps || !argmax || !sample || !entropy) return DRS_ERR_INVALID_ARG;
    if (probs_dtype != DRS_PROBS_NONE && probs_dtype != DRS_PROBS_BF16 &&
        probs_dtype != DRS_PROBS_FP16)
        return DRS_ERR_INVALID_ARG;
    if ((probs_dtype == DRS_PROBS_NONE) != (probs == nullptr)) return DRS_ERR_INVALID_ARG;
    if (probs && probs_row_stride < vocab) return DRS_ERR_INVALID_ARG;
    if (!aligned(logits, 4) || !aligned(probs, 2)) return DRS_ERR_INVALID_ARG;
    return DRS_OK;
}

// Top-k of the converged rows into a workspace laid out as: the split
// kernels' workspace (the hard-row list first), the exact kernel's records.
drs_status run_topk(RowCall c, void* workspace, cudaStream_t stream) {
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    const int32_t* hard = reinterpret_cast<const int32_t*>(ws);
    void* exact_ws = ws + split_workspace_bytes(c.rows, c.vocab, c.k > split_max_k() ? 0 : c.k, 1);
    if (c.k > split_max_k()) {
        // larger k: the row statistics alone, then the exact kernel on every
        // converged row
        if (c.stats) {
            RowCall s = c;
            s.k = 0;
            s.keep = nullptr;
            const drs_status st = split_rows(s, workspace, stream);
            if (st != DRS_OK) return st;
        }
        return exact_topk(c.logits, c.rows, c.vocab, c.row_stride, c.row0, c.temps, c.canvas_len,
                          c.keep, nullptr, c.k, c.out_ids, c.out_lp, exact_ws, stream);
    }
    const drs_status st = split_rows(c, workspace, stream);
    if (st != DRS_OK) return st;
    // the rows the split kernels left (no threshold, or too many candidates)
    return exact_topk(c.logits, c.rows, c.vocab, c.row_stride, c.row0, c.temps, c.canvas_len,
                      c.keep, hard, c.k, c.out_ids, c.out_lp, exact_ws, stream);
}

}  // namespace
}  // namespace drs

int drs::take_injected_fault() { return drs::g_inject_fault.exchange(0); }

extern "C" void drs_test_inject_fault(int code) { drs::g_inject_fault.store(code); }

bool drs::two_pass_forced() { return drs::g_two_pass.load() != 0; }

extern "C" void drs_test_two_pass(int on) { drs::g_two_pass.store(on ? 1 : 0); }

extern "C" drs_status drs_row_split_plan(int64_t rows, int64_t vocab, int32_t k, int32_t n_seeds,
                                         int probs_dtype, int32_t stats, int64_t* cluster_rows,
                                         int32_t* cluster_size,
                                         int32_t* clusters, int32_t* free_sms) {
    if (!cluster_rows || !cluster_size || !clusters || !free_sms) return DRS_ERR_INVALID_ARG;
    if (rows < 0 || vocab < 1 || n_seeds < 1 || probs_dtype < 0 || probs_dtype > 2) return DRS_ERR_INVALID_ARG;
    *cluster_rows = 0;
    *cluster_size = 0;
    *clusters = 0;
    *free_sms = 0;
    if (rows == 0) return DRS_OK;
    drs::split_plan_query(rows, vocab, k, n_seeds, true, probs_dtype, stats != 0, cluster_rows, cluster_size,
                          clusters, free_sms);
    return DRS_OK;
}

extern "C" size_t drs_row_stats_workspace_bytes(int64_t rows, int64_t vocab) {
    if (rows < 0 || vocab < 1) return 0;
    return drs::split_workspace_bytes(rows, vocab, 0, 1);
}

extern "C" drs_status drs_row_stats(const float* logits, int64_t rows, int64_t vocab,
                                    int64_t row_stride, const float* temps,
                                    int64_t canvas_len, uint64_t seed, int64_t row0,
                                    int64_t* argmax, int64_t* sample, float* entropy,
                                    drs_probs_dtype probs_dtype, void* probs,
                                    int64_t probs_row_stride, void* workspace,
                                    size_t workspace_bytes, void* stream) {
    using namespace drs;
    const drs_status chk = check_stats_args(logits, rows, vocab, row_stride, temps, canvas_len,
                                            row0, argmax, sample, entropy, probs_dtype, probs,
                                            probs_row_stride);
    if (chk != DRS_OK) return chk;
    if (rows == 0) return DRS_OK;
    const size_t need = drs_row_stats_workspace_bytes(rows, vocab);
    if (!workspace || workspace_bytes < need || !aligned(workspace, kWorkspaceAlign))
        return DRS_ERR_INVALID_ARG;
    RowCall c{logits, rows, vocab, row_stride, temps, canvas_len, seed, nullptr, 1, row0, argmax,
              sample, entropy, probs_dtype, probs, probs_row_stride, nullptr, 0, nullptr, nullptr,
              true};
    return split_rows(c, workspace, static_cast<cudaStream_t>(stream));
}

extern "C" size_t drs_row_stats_seeds_workspace_bytes(int64_t rows, int64_t vocab,
                                                     int32_t n_seeds) {
    if (rows < 0 || vocab < 1 || n_seeds < 1 || n_seeds > drs::split_max_seeds()) return 0;
    return drs::split_workspace_bytes(rows, vocab, 0, n_seeds);
}

extern "C" drs_status drs_row_stats_seeds(const float* logits, int64_t rows, int64_t vocab,
                                          int64_t row_stride, const float* temps,
                                          int64_t canvas_len, const uint64_t* seeds,
                                          int32_t n_seeds, int64_t row0, int64_t* argmax,
                                          int64_t* samples, float* entropy,
                                          drs_probs_dtype probs_dtype, void* probs,
                                          int64_t probs_row_stride, void* workspace,
                                          size_t workspace_bytes, void* stream) {
    using namespace drs;
    const drs_status chk = check_stats_args(logits, rows, vocab, row_stride, temps, canvas_len,
                                            row0, argmax, samples, entropy, probs_dtype, probs,
                                            probs_row_stride);
    if (chk != DRS_OK) return chk;
    if (!seeds || n_seeds < 1 || n_seeds > split_max_seeds()) return DRS_ERR_INVALID_ARG;
    if (rows == 0) return DRS_OK;
    const size_t need = drs_row_stats_seeds_workspace_bytes(rows, vocab, n_seeds);
    if (!workspace || workspace_bytes < need || !aligned(workspace, kWorkspaceAlign))
        return DRS_ERR_INVALID_ARG;
    RowCall c{logits, rows, vocab, row_stride, temps, canvas_len, seeds[0], seeds, n_seeds, row0,
              argmax, samples, entropy, probs_dtype, probs, probs_row_stride, nullptr, 0, nullptr,
              nullptr, true};
    return split_rows(c, workspace, static_cast<cudaStream_t>(stream));
}

extern "C" size_t drs_row_stats_topk_workspace_bytes(int64_t rows, int64_t vocab, int32_t k) {
    if (k <= 0 || rows < 0 || vocab < 1) return 0;
    const int32_t ks = k > drs::split_max_k() ? 0 : k;
    return drs::split_workspace_bytes(rows, vocab, ks, 1) + drs::exact_topk_workspace_bytes(k);
}

extern "C" drs_status drs_row_stats_topk(const float* logits, int64_t rows, int64_t vocab,
                                         int64_t row_stride, const float* temps,
                                         int64_t canvas_len, uint64_t seed, int64_t row0,
                                         int64_t* argmax, int64_t* sample, float* entropy,
                                         drs_probs_dtype probs_dtype, void* probs,
                                         int64_t probs_row_stride, const uint8_t* keep, int32_t k,
                                         int32_t* out_ids, float* out_logprobs, void* workspace,
                                         size_t workspace_bytes, void* stream) {
    using namespace drs;
    const drs_status chk = check_stats_args(logits, rows, vocab, row_stride, temps, canvas_len,
                                            row0, argmax, sample, entropy, probs_dtype, probs,
                                            probs_row_stride);
    if (chk != DRS_OK) return chk;
    if (k < 0 || k > vocab || k > exact_topk_max_k()) return DRS_ERR_INVALID_ARG;
    if (k > 0 && (!keep || !out_ids || !out_logprobs)) return DRS_ERR_INVALID_ARG;
    if (rows == 0) return DRS_OK;
    if (k == 0)
        return drs_row_stats(logits, rows, vocab, row_stride, temps, canvas_len, seed, row0,
                             argmax, sample, entropy, probs_dtype, probs, probs_row_stride,
                             workspace, workspace_bytes, stream);
    const size_t need = drs_row_stats_topk_workspace_bytes(rows, vocab, k);
    if (!workspace || workspace_bytes < need || !aligned(workspace, kWorkspaceAlign))
        return DRS_ERR_INVALID_ARG;
    RowCall c{logits, rows, vocab, row_stride, temps, canvas_len, seed, nullptr, 1, row0, argmax,
              sample, entropy, probs_dtype, probs, probs_row_stride, keep, k, out_ids, out_logprobs,
              true};
    return run_topk(c, workspace, static_cast<cudaStream_t>(stream));
}

extern "C" size_t drs_topk_workspace_bytes(int64_t rows, int64_t vocab, int32_t k) {
    return drs_row_stats_topk_workspace_bytes(rows, vocab, k);
}

extern "C" drs_status drs_topk_logprobs(const float* logits, int64_t rows, int64_t vocab,
                                        int64_t row_stride, const float* temps,
                                        int64_t canvas_len, const uint8_t* keep, int32_t k,
                                        int32_t* out_ids, float* out_logprobs, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    using namespace drs;
    if (rows < 0 || canvas_len < 1 || k < 0) return DRS_ERR_INVALID_ARG;
    if (vocab < 1 || row_stride < vocab) return DRS_ERR_INVALID_ARG;
    if (vocab > DRS_MAX_VOCAB) return DRS_ERR_UNSUPPORTED;
    if (k > vocab || k > exact_topk_max_k()) return DRS_ERR_INVALID_ARG;
    if (rows % canvas_len != 0) return DRS_ERR_INVALID_ARG;
    if (k == 0 || rows == 0) return DRS_OK;
    if (!logits || !temps || !keep || !out_ids || !out_logprobs) return DRS_ERR_INVALID_ARG;
    if (!aligned(logits, 4)) return DRS_ERR_INVALID_ARG;
    const size_t need = drs_topk_workspace_bytes(rows, vocab, k);
    if (!workspace || workspace_bytes < need || !aligned(workspace, kWorkspaceAlign))
        return DRS_ERR_INVALID_ARG;
    RowCall c{logits, rows, vocab, row_stride, temps, canvas_len, 0, nullptr, 1, 0, nullptr,
              nullptr, nullptr, DRS_PROBS_NONE, nullptr, 0, keep, k, out_ids, out_logprobs, false};
    return run_topk(c, workspace, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// drs_row_stats_noalloc: drs_row_stats with its workspace in a fixed device
// array of this library instead of a caller buffer.
//
// Some callers cannot hand the library a workspace: plugin interfaces of
// inference runtimes that pass only input and output buffers at enqueue
// time, or code that must not call cudaMalloc because it synchronises the
// device or draws on a memory budget fixed at start-up. For them the row
// kernels' records live in g_noalloc_workspace below: every GPU that loads
// the library holds these bytes until the process exits, and all calls on a
// device share them. A call whose rows need more runs in batches of rows
// that fit.

namespace {

constexpr size_t kNoallocWorkspaceBytes = static_cast<size_t>(640) * 1024;
static __device__ __align__(256) unsigned char g_noalloc_workspace[kNoallocWorkspaceBytes];

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[64] = {};

// Device address of g_noalloc_workspace on the current device. In host code
// the array's name is a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
void* noalloc_workspace(drs_status* status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *status = DRS_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_workspace);
        if (e != cudaSuccess || !ptr) {
            *status = DRS_ERR_CUDA;
            return nullptr;
        }
        g_noalloc_ptr[dev] = ptr;
    }
    *status = DRS_OK;
    return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" drs_status drs_row_stats_noalloc(const float* logits, int64_t rows, int64_t vocab,
                                            int64_t row_stride, const float* temps,
                                            int64_t canvas_len, uint64_t seed, int64_t row0,
                                            int64_t* argmax, int64_t* sample, float* entropy,
                                            drs_probs_dtype probs_dtype, void* probs,
                                            int64_t probs_row_stride, void* stream) {
    const drs_status chk = drs::check_stats_args(logits, rows, vocab, row_stride, temps,
                                                 canvas_len, row0, argmax, sample, entropy,
                                                 probs_dtype, probs, probs_row_stride);
    if (chk != DRS_OK) return chk;
    if (rows == 0) return DRS_OK;
    // rows in batches whose workspace fits the array (one row always does)
    int64_t batch = rows;
    while (batch > 1 && drs_row_stats_workspace_bytes(batch, vocab) > kNoallocWorkspaceBytes)
        batch = (batch + 1) / 2;
    if (drs_row_stats_workspace_bytes(batch, vocab) > kNoallocWorkspaceBytes)
        return DRS_ERR_UNSUPPORTED;
    drs_status st = DRS_OK;
    void* ws = noalloc_workspace(&st);
    if (!ws) return st;
    const size_t pbytes = probs_dtype == DRS_PROBS_NONE ? 0 : 2;
    for (int64_t r = 0; r < rows; r += batch) {
        const int64_t n = rows - r < batch ? rows - r : batch;
        void* pr = probs ? static_cast<unsigned char*>(probs) +
                               static_cast<size_t>(r) * static_cast<size_t>(probs_row_stride) * pbytes
                         : nullptr;
        st = drs_row_stats(logits + r * row_stride, n, vocab, row_stride, temps, canvas_len, seed,
                           row0 + r, argmax + r, sample + r, entropy + r, probs_dtype, pr,
                           probs_row_stride, ws, kNoallocWorkspaceBytes, stream);
        if (st != DRS_OK) return st;
    }
    return DRS_OK;
}
