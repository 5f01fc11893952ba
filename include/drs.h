/*
 * drs.h -- C ABI of libdrs, the GB300 (sm_103a) implementation of the
 * DiffusionGemma per-row sampler statistics.
 *
 * The operations follow the page "vllm.model_executor.models.
 * diffusion_gemma_sampler": the module docstring (argmax, Gumbel-max sample,
 * softmax entropy and the softmax in the model dtype, the noise drawn inline),
 * sample_row_stats and its PyTorch definition sample_row_stats_reference,
 * and stash_converged_logprobs / _lp_topk_kernel (top-k logprobs of the rows
 * of converged slots, keys ordered by value then by lower index).
 *
 * Conventions for every entry point:
 *   - Array arguments are DEVICE pointers owned by the caller, unless stated
 *     otherwise. The library allocates no device memory in any call.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream). Results are ready when the
 *     stream is.
 *   - Host-side argument checks return DRS_ERR_INVALID_ARG without
 *     launching anything. Launch failures return DRS_ERR_CUDA. A device-side
 *     wait that runs out of time makes the kernel skip its remaining writes
 *     and raise a device flag, read with drs_get_device_error().
 *   - The library cannot check the length of device arrays; the caller
 *     guarantees the sizes stated below.
 *   - Not thread-safe for concurrent calls that share one workspace.
 */
#ifndef DRS_H_
#define DRS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum drs_status {
    DRS_OK = 0,
    DRS_ERR_INVALID_ARG = -1,
    DRS_ERR_UNSUPPORTED = -2,
    DRS_ERR_CUDA = -3,
    DRS_ERR_DEVICE_TIMEOUT = -4
} drs_status;

typedef enum drs_probs_dtype {
    DRS_PROBS_NONE = 0,
    DRS_PROBS_BF16 = 1,
    DRS_PROBS_FP16 = 2
} drs_probs_dtype;

/* Largest vocabulary (row length) the kernels accept (2^21). */
#define DRS_MAX_VOCAB 2097152

/*
 * Bytes of device workspace drs_row_stats needs (at least 256-byte aligned,
 * contents arbitrary: each call clears the counters it uses with an
 * asynchronous memset on its stream before its kernels run). The workspace
 * carries the row lists and the per-tile and per-row records through which
 * the kernels of one call pass their partial results: about 4.6 KiB per row
 * of 262144 columns, growing with rows and vocab. One workspace must not be
 * used by two calls that can run at the same time.
 */
size_t drs_row_stats_workspace_bytes(int64_t rows, int64_t vocab);

/*
 * Per-row statistics of temperature-scaled logits (sample_row_stats and
 * sample_row_stats_reference on the page above).
 *
 *   logits      fp32 [rows, vocab], row i at logits + i * row_stride, unit
 *               column stride. row_stride >= vocab; the columns between
 *               vocab and row_stride are never read.
 *   row0        global index of the first row (>= 0). Row i of this call
 *               is global row row0 + i: it keys the noise and picks the
 *               temperature, so a batch split over several calls or GPUs
 *               gives the results of one call. 0 for a whole batch.
 *   temps       fp32 [ceil((row0 + rows) / canvas_len)], one per slot of the
 *               whole batch; global row r uses T = temps[r / canvas_len].
 *               The scaled logit is the IEEE fp32
 *               quotient x / max(T, 1e-10f). T > 0 draws Gumbel noise; T <= 0
 *               is greedy (sample = argmax). NaN temperatures, NaN or +inf
 *               logits are not supported; -inf logits are.
 *   seed        noise key. The noise of (global row, col) is Philox4x32-10
 *               with key
 *               (lo32(seed), hi32(seed)) and counter (lo32(col/4),
 *               hi32(col/4), lo32(row), hi32(row)), word col % 4, mapped to
 *               u = max((word >> 8) * 2^-24, 1e-20f); g = -log(-log u). The
 *               same function is exposed by drs_philox_gumbel.
 *   argmax      int64 [rows]: lowest column of the largest scaled logit.
 *   sample      int64 [rows]: lowest column of the largest scaled logit + g.
 *   entropy     fp32 [rows]: entropy of softmax(scaled); -inf columns drop
 *               out; a row that is -inf everywhere has entropy 0.
 *   probs       probs_dtype NONE: must be NULL. BF16/FP16: 16-bit
 *               [rows, vocab] with row stride probs_row_stride >= vocab
 *               (elements), softmax(scaled) rounded to nearest even.
 *   workspace   device scratch of drs_row_stats_workspace_bytes(rows, vocab)
 *               bytes; may be NULL only when that function returns 0.
 *
 * rows == 0 returns DRS_OK without launching. vocab must be in
 * [1, DRS_MAX_VOCAB]; canvas_len >= 1.
 */
drs_status drs_row_stats(const float *logits, int64_t rows, int64_t vocab,
                         int64_t row_stride, const float *temps,
                         int64_t canvas_len, uint64_t seed, int64_t row0,
                         int64_t *argmax,
                         int64_t *sample, float *entropy,
                         drs_probs_dtype probs_dtype, void *probs,
                         int64_t probs_row_stride, void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * drs_row_stats without a caller workspace. The page has no counterpart:
 * this entry point exists for callers that cannot allocate device memory
 * for the library -- plugin interfaces that hand over only input and
 * output buffers at enqueue time, or code that must not call cudaMalloc
 * (it can synchronise the device, or the memory budget is fixed at
 * start-up). Arguments, results and errors are those of drs_row_stats.
 *
 * The kernels' records live in a fixed device array inside the library
 * (640 KiB; every GPU that loads the library holds it until the process
 * exits). A call whose rows need a larger workspace runs in batches of rows
 * that fit, one after the other on the stream (at most 137 rows of 262144
 * columns per batch). The call allocates nothing. Its
 * first call on a device looks up the array's device address (with that
 * device current) and caches it; make that first call before any stream
 * capture. All calls on a device share the array: two calls that can run
 * at the same time on the GPU (different streams, overlapping) race and
 * corrupt each other's results. Each call resets the list counters at the
 * start of the array (an asynchronous memset on its stream) before its
 * kernels run; every other record in the array is written before it is read
 * within the same call, so what an earlier call left there is never used.
 * The cached address belongs to the device's CUDA context: after
 * cudaDeviceReset (or anything else that destroys the primary context) the
 * library must be unloaded and loaded again before this entry point is
 * called on that device.
 */
drs_status drs_row_stats_noalloc(const float *logits, int64_t rows, int64_t vocab,
                                 int64_t row_stride, const float *temps,
                                 int64_t canvas_len, uint64_t seed, int64_t row0,
                                 int64_t *argmax, int64_t *sample, float *entropy,
                                 drs_probs_dtype probs_dtype, void *probs,
                                 int64_t probs_row_stride, void *stream);

/*
 * Bytes of device workspace drs_row_stats_seeds needs for n_seeds seeds
 * (1 <= n_seeds <= 8; 0 otherwise). Same alignment and sharing rules as the
 * row-stats workspace.
 */
size_t drs_row_stats_seeds_workspace_bytes(int64_t rows, int64_t vocab, int32_t n_seeds);

/*
 * drs_row_stats for several noise seeds in one call: the argmax, entropy and
 * probabilities once, and a Gumbel-max sample per seed, from the same two
 * passes over the logits (the race of each seed runs on the tile already in
 * shared memory). Every argument of drs_row_stats has its meaning there;
 * in addition:
 *
 *   seeds       HOST uint64 [n_seeds], 1 <= n_seeds <= 8: the noise keys.
 *   samples     int64 [n_seeds, rows]: samples + s * rows is the sample of
 *               every row under seeds[s] (what drs_row_stats gives with that
 *               seed).
 *   workspace   drs_row_stats_seeds_workspace_bytes(rows, vocab, n_seeds).
 *
 * Returns DRS_ERR_INVALID_ARG for a null seeds array or n_seeds outside
 * [1, 8], otherwise as drs_row_stats.
 */
drs_status drs_row_stats_seeds(const float *logits, int64_t rows, int64_t vocab,
                               int64_t row_stride, const float *temps,
                               int64_t canvas_len, const uint64_t *seeds,
                               int32_t n_seeds, int64_t row0, int64_t *argmax,
                               int64_t *samples, float *entropy,
                               drs_probs_dtype probs_dtype, void *probs,
                               int64_t probs_row_stride, void *workspace,
                               size_t workspace_bytes, void *stream);

/*
 * Bytes of device workspace drs_row_stats_topk needs for k > 0 (256-byte
 * aligned, contents arbitrary: each call clears what it uses with
 * asynchronous memsets on its stream). 0 for k <= 0, where the call needs
 * drs_row_stats_workspace_bytes() instead. Same sharing rule as the
 * row-stats workspace.
 */
size_t drs_row_stats_topk_workspace_bytes(int64_t rows, int64_t vocab, int32_t k);

/*
 * drs_row_stats and the top-k logprobs of the rows of converged slots from
 * the same read of the logits (stash_converged_logprobs /
 * _lp_topk_kernel on the page above, whose stash reads the kept rows again
 * in a kernel of its own). Every argument of drs_row_stats has its meaning
 * there; in addition:
 *
 *   keep        uint8 [ceil((row0 + rows) / canvas_len)], one per slot of
 *               the whole batch like temps: global row r is converged when
 *               keep[r / canvas_len] != 0.
 *   k           0 <= k <= min(vocab, 1024); k == 0 is drs_row_stats (with
 *               its workspace size).
 *   out_ids     int32 [rows, k]: for a converged row, the columns of the k
 *               largest scaled logits, ordered by value and then by lower
 *               column (-0.0 equals +0.0). Rows of other slots are not
 *               written.
 *   out_logprobs fp32 [rows, k]: scaled - max - log(sum exp(scaled - max))
 *               of those columns (NaN for a row that is -inf everywhere).
 *   workspace   drs_row_stats_topk_workspace_bytes(rows, vocab, k) bytes.
 *
 * For k <= 64 the top-k candidates come out of the row statistics' own read
 * of the logits: in the cluster kernel the threshold from the CTAs' parts
 * (distributed shared memory) and the candidates from the row held in shared
 * memory; in the two passes the threshold from the first and the candidates
 * in the second. Rows whose candidates overflow the fixed lists (many equal
 * values) or that have no threshold are finished by the exact top-k kernel
 * on the same stream, which reads only those rows. For k > 64 the row
 * statistics and the exact top-k kernel run one after the other.
 */
drs_status drs_row_stats_topk(const float *logits, int64_t rows, int64_t vocab,
                              int64_t row_stride, const float *temps,
                              int64_t canvas_len, uint64_t seed, int64_t row0,
                              int64_t *argmax, int64_t *sample, float *entropy,
                              drs_probs_dtype probs_dtype, void *probs,
                              int64_t probs_row_stride, const uint8_t *keep,
                              int32_t k, int32_t *out_ids, float *out_logprobs,
                              void *workspace, size_t workspace_bytes,
                              void *stream);

/*
 * Bytes of device workspace drs_topk_logprobs needs (256-byte aligned,
 * contents arbitrary). Same sharing rule as the row-stats workspace.
 */
size_t drs_topk_workspace_bytes(int64_t rows, int64_t vocab, int32_t k);

/*
 * Top-k logprobs of the rows of converged slots (stash_converged_logprobs
 * and _lp_topk_kernel on the page above).
 *
 *   logits, rows, vocab, row_stride, temps, canvas_len: as drs_row_stats;
 *               rows must be a multiple of canvas_len.
 *   keep        uint8 [rows / canvas_len]: slot n is converged when
 *               keep[n] != 0. Rows of other slots are skipped and their
 *               outputs are not written.
 *   k           0 <= k <= min(vocab, 1024); k == 0 does nothing.
 *   out_ids     int32 [rows, k]: for a kept row, the columns of the k
 *               largest scaled logits, ordered by value and then by lower
 *               column (-0.0 equals +0.0).
 *   out_logprobs fp32 [rows, k]: scaled - max - log(sum exp(scaled - max))
 *               of those columns (NaN for a row that is -inf everywhere).
 *
 * For k <= 64 this runs the kernels of drs_row_stats_topk with the row
 * statistics off (rows of unconverged slots are not read); larger k, and
 * rows with many equal values, use the exact top-k kernel.
 */
drs_status drs_topk_logprobs(const float *logits, int64_t rows, int64_t vocab,
                             int64_t row_stride, const float *temps,
                             int64_t canvas_len, const uint8_t *keep,
                             int32_t k, int32_t *out_ids, float *out_logprobs,
                             void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * The sampler's noise, materialised (the generator of drs_row_stats).
 * Page "vllm.model_executor.models.diffusion_gemma_sampler",
 * sample_row_stats_reference: the Gumbel noise -log(-log u) of a uniform u
 * drawn like rand_like(...) and clamped below at 1e-20; the page's kernel
 * takes a seed, and the uniform is drawn here by Philox4x32-10 (Salmon,
 * Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3",
 * SC'11) keyed and laid out as the `seed` argument of drs_row_stats states.
 * For r in [0, rows), c in [0, vocab): out_bits[r * vocab + c] is the
 * Philox word of (row0 + r, c) and out_gumbel[r * vocab + c] the fp32
 * -log(-log u) of it, u = max((word >> 8) * 2^-24, 1e-20f). Either output
 * may be NULL; rows == 0 is a no-op. Outputs are caller-owned device
 * memory; invalid sizes return DRS_ERR_INVALID_ARG before any launch.
 */
drs_status drs_philox_gumbel(uint64_t seed, int64_t row0, int64_t rows,
                             int64_t vocab, uint32_t *out_bits,
                             float *out_gumbel, void *stream);

/*
 * The temperature-scaled logits of sample_row_stats_reference (page above):
 * out[i] = logits[i] / max(temp, 1e-10f) for i < n, the IEEE fp32 quotient
 * rounded to nearest even, computed by the same routine the row kernels use
 * (+-inf map to themselves). logits and out: device fp32 [n], 4-byte
 * aligned; they may be the same array. n == 0 is a no-op.
 */
drs_status drs_scaled_logits(const float *logits, int64_t n, float temp,
                             float *out, void *stream);

/*
 * Test hook for the failure path (not for production use). code != 0: in
 * the next row-statistics call of this process, CTA 0 of the first pass
 * never fills its first shared-memory stage. Its warps' bounded waits on the
 * stage run out (about 1 s), the CTA stops and raises the device flag that
 * drs_get_device_error reports; the call's results are not valid, the CUDA
 * context stays usable. The hook resets itself after one call; code 0
 * clears it.
 */
void drs_test_inject_fault(int code);

/*
 * Test hook (not for production use). on != 0: from now on every
 * row-statistics call of this process takes the two streaming passes over
 * the logits (list of rows, pass 1, merge, pass 2, finish) even where the
 * one-read cluster kernel would take it (rows that start 16-byte aligned,
 * vocab a multiple of 4 and at most 262144, one seed, k <= 64). Results are
 * the same within the tolerances of the method; the hook exists so that
 * both implementations can be tested and timed on the same inputs. on == 0
 * restores the automatic choice.
 */
void drs_test_two_pass(int on);

/*
 * Introspection (not part of the sampler): how a row-statistics call of
 * these sizes shares its rows on the current device. Calls whose rows start
 * 16-byte aligned, with vocab a multiple of 4 and at most 262144, one seed
 * and k <= 64 read each row once, split over the CTAs of a thread-block
 * cluster (*cluster_size CTAs per row, *clusters clusters resident at once,
 * one CTA per SM); such clusters fit only some of the GPU's SM groups, and on
 * large calls the *free_sms SMs they leave run the two streaming passes over
 * the tail of the call's row list at the same time. *cluster_rows is the
 * head of a list of `rows` entries; a call whose list is shorter (a top-k
 * call lists the rows of kept slots only) divides it in the same proportion
 * on the device. Other calls take the two passes alone: *cluster_rows, *cluster_size,
 * *clusters and *free_sms are then 0. probs_dtype: a drs_probs_dtype value;
 * stats: nonzero for the calls that compute the row statistics
 * (drs_row_stats, drs_row_stats_topk), 0 for the top-k calls
 * (drs_topk_logprobs, the stash). Top-k calls take no cluster kernel: they
 * read each row once in the first streaming pass and then only the columns
 * of the row's warps whose max reaches its top-k threshold (all outputs 0).
 * All outputs are HOST pointers. Returns DRS_OK, or DRS_ERR_INVALID_ARG for a
 * null pointer or sizes out of range.
 */
drs_status drs_row_split_plan(int64_t rows, int64_t vocab, int32_t k, int32_t n_seeds,
                              int probs_dtype, int32_t stats, int64_t *cluster_rows,
                              int32_t *cluster_size, int32_t *clusters, int32_t *free_sms);

/*
 * Measurement hook (not part of the sampler). enable != 0: from now on every
 * row-statistics call on the current device (drs_row_stats, its no-alloc and
 * top-k variants, drs_topk_logprobs for k <= 64) records a CUDA event on
 * its stream before each of six kernel slots (list of rows, pass 1, merge,
 * pass 2, cluster, finish) and after the last; the slots a call does not
 * launch (the two passes or the cluster kernel) measure about 0, and a
 * top-k call's finish slot times its gather (split_gather). The count
 * of recorded calls restarts at 0. enable == 0 stops recording. The events
 * of the last 64 calls are kept. Returns DRS_OK or DRS_ERR_CUDA (event
 * creation failed).
 */
drs_status drs_kernel_timing(int enable);

/*
 * Average device time in ms of each kernel slot of the recorded calls (see
 * drs_kernel_timing), in the order above, into the HOST array avg_ms[n]
 * (entries past the sixth are 0); *calls (HOST) receives the number of
 * calls averaged (at most 64). Waits for the recorded events. Returns
 * DRS_OK, DRS_ERR_INVALID_ARG (null pointer, n < 0) or DRS_ERR_CUDA.
 */
drs_status drs_kernel_times(float *avg_ms, int32_t n, int32_t *calls);

/*
 * Bytes of device workspace drs_stash_converged_logprobs needs (256-byte
 * aligned, contents arbitrary); 0 for arguments outside its ranges
 * (num_topk in [0, 1024]).
 */
size_t drs_stash_workspace_bytes(int64_t requests, int64_t canvas_len, int64_t vocab,
                                 int32_t num_topk);

/*
 * The stash of converged requests' logprobs (stash_converged_logprobs on
 * the page above, its docstring). Request j < requests owns logits rows
 * src[j] * canvas_len + p for p < valid[j], scaled by
 * max(temps[j], 1e-10). Where keep[j] != 0, stash row
 * slots[j] * canvas_len + p of the outputs receives `width` columns of
 * (id, value):
 *   column 0        the argmax of the scaled row (lowest column of the max);
 *   then            token_ids[j * ids_stride + c] for c < n_j =
 *                   min(num_token_ids[j], ids_stride) when token_ids is
 *                   given and n_j > 0 (a request's list holds ids_stride
 *                   ids; a larger count reads no further), else
 *                   the num_topk largest (value descending, lower column
 *                   first);
 *   then            id 0 with value -inf, up to `width`.
 * value: the logprob s - max - log(sum over the row of e^(s - max)) (NaN
 * when the row is -inf everywhere), or the scaled logit s itself when
 * logits_mode != 0; NaN for a token id outside [0, vocab).
 * out_ranks[stash row]: 1 + the number of columns whose scaled logit
 * exceeds column 0's (column 0 is the argmax, so 1).
 *
 *   logits          fp32, row r at logits + r * row_stride, r < logits_rows.
 *   src, slots, valid, num_token_ids   int32 [requests] (num_token_ids may
 *                   be null without token_ids).
 *   keep            uint8 [requests]; temps fp32 [requests].
 *   token_ids       null, or int32 [requests, ids_stride].
 *   out_ids         int32 [out_slots * canvas_len, width]; out_logprobs
 *                   fp32 and out_ranks int32 [out_slots * canvas_len] alike.
 *                   Rows of requests not kept, positions p >= valid[j], and
 *                   rows whose logits row or stash row falls outside
 *                   logits_rows or out_slots are not touched.
 *   workspace       drs_stash_workspace_bytes(requests, canvas_len, vocab,
 *                   num_topk) bytes.
 * The slots of kept requests must be distinct: two requests writing one
 * stash row race (which one lands is not defined).
 * All pointers are device memory owned by the caller; asynchronous on
 * `stream`. Returns DRS_ERR_INVALID_ARG for a null required pointer,
 * negative sizes, row_stride < vocab, num_topk outside [0, min(vocab,
 * 1024)], width < num_topk + 1, token_ids without num_token_ids or with
 * ids_stride < 1, or a small or unaligned workspace;
 * DRS_ERR_UNSUPPORTED for vocab > DRS_MAX_VOCAB or more than 2^31 - 1
 * stash rows; requests == 0 is a no-op.
 */
drs_status drs_stash_converged_logprobs(const float *logits, int64_t logits_rows, int64_t vocab,
                                        int64_t row_stride, int64_t canvas_len, int64_t requests,
                                        const int32_t *src, const int32_t *slots,
                                        const uint8_t *keep, const int32_t *valid,
                                        const float *temps, int32_t num_topk,
                                        const int32_t *num_token_ids, const int32_t *token_ids,
                                        int64_t ids_stride, int64_t out_slots, int32_t width,
                                        int32_t *out_ids, float *out_logprobs,
                                        int32_t *out_ranks, int logits_mode, void *workspace,
                                        size_t workspace_bytes, void *stream);

/* Static, human-readable name of a status code. */
const char *drs_status_string(drs_status s);

/*
 * Synchronise `stream`, then read and clear the device flag raised by a
 * kernel whose bounded wait ran out of time on the current device.
 * Returns DRS_OK, DRS_ERR_DEVICE_TIMEOUT or DRS_ERR_CUDA.
 */
drs_status drs_get_device_error(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DRS_H_ */
