/*
 * specverify.h -- libspecverify: batched draft-token verification by modified
 * rejection sampling, on one NVIDIA GB300 (sm_103a).
 *
 * The operation (defined on the pages this library follows):
 *  - tech-tldr.com "投機的デコーディングとドラフトモデル", section
 *    受理判定の数理：修正版棄却サンプリング: keep proposal x_i when a uniform
 *    r in [0,1) satisfies r < min(1, p(x_i)/q(x_i)); at the first failure stop
 *    and draw one token from normalize(max(0, p - q)).
 *  - r-jc.jp "LLM推論の高速化｜KVキャッシュと投機的デコーディングを自作で実測",
 *    section 投機的デコーディングとは（speculative decoding の仕組み): per
 *    position p = softmax(target logits / T), q = softmax(draft logits / T);
 *    ordered tests, first-rejection break; after the loop row nacc supplies
 *    the residual (a rejection happened) or p itself (all accepted: the bonus
 *    token); one inverse-CDF draw; the caller then truncates its KV cache to
 *    base + 1 + nacc.  Section 投機的デコーディングを実装して受理率と速度を実測:
 *    at temperature 0 a proposal is kept iff it equals the target argmax.
 *  - issoh.co.jp "Speculative Decoding（投機的デコーディング）とは？…",
 *    section 受理・棄却の規則と出力分布が変わらない理由, steps 1-5.
 *
 * Conventions shared by every entry point
 *  - Layouts are row-major and contiguous:
 *      target_logits [B][Kmax+1][V], draft_logits [B][Kmax][V] (same dtype),
 *      draft_tokens [B][Kmax] int32, uniforms [B][Kmax+1] float32,
 *      temperature [B] float32, out_tokens [B][Kmax+1] int32,
 *      out_num_accepted [B] int32,
 *    where Kmax = max_b K[b] is computed from the host array K.
 *  - Uniform slots: uniforms[b][i] for i < K[b] is the accept test of
 *    position i; uniforms[b][K[b]] is the final draw (resample or bonus).
 *    Slots past K[b] are never read.  Greedy sequences read no uniforms.
 *  - temperature[b] == 0 selects greedy verification for sequence b; any
 *    other usable value (finite, >= FLT_MIN) selects sampling at that T.
 *  - Outputs: out_tokens[b][j] = draft_tokens[b][j] for j < n_b, the drawn
 *    token at j = n_b, -1 after it; out_num_accepted[b] = n_b.  The caller
 *    sets its KV length to base + 1 + n_b.
 *  - Device-data errors never trap: a NaN or +inf logit, a row with no finite
 *    entry, an unusable temperature, a token outside [0, V) or a uniform
 *    outside [0,1) met on the path the method walks makes that sequence's
 *    out_num_accepted -1 and its out_tokens row all -1.  Rows after the first
 *    rejection are never read, so their contents cannot affect the result.
 *  - Host-detectable argument errors return synchronously before any work is
 *    queued.  Launches are asynchronous on `stream`; nothing synchronises the
 *    device except spec_verify_host and sv_workspace_errors, which say so.
 *  - All buffers are owned by the caller.  Device pointers must belong to
 *    the current device.  16-byte-aligned logits with V*sizeof(elem) a
 *    multiple of 16 take the bulk-copy (TMA) path; anything else is still
 *    accepted and read with element loads.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SV_ABI_VERSION 5
/* Largest per-sequence draft count: one warp ballot covers the accept bits. */
#define SV_K_MAX 32

typedef enum {
    SV_OK = 0,
    SV_ERR_INVALID_ARG = 1,   /* bad pointer, size, K[b] or dtype; nothing queued */
    SV_ERR_CUDA = 2,          /* a CUDA runtime call failed */
    SV_ERR_UNSUPPORTED = 3,   /* V beyond sv_max_vocab(dtype) */
    SV_ERR_NO_MEMORY = 4,     /* workspace too small, or stream-ordered allocation failed */
    SV_ERR_TIMEOUT = 5        /* a bounded device-side wait gave up (see sv_workspace_errors) */
} sv_status;

typedef enum { SV_DTYPE_F32 = 0, SV_DTYPE_BF16 = 1 } sv_dtype;

/*
 * Optional per-position diagnostics (device pointers; each may be NULL).
 *   p_x, q_x    [B][Kmax] float32: p_i(x_i) and q_i(x_i) at every draft
 *               position i < K[b] of a sampling sequence; NaN elsewhere
 *               (greedy sequence, i >= K[b], unusable row or token).
 *   resid_mass  [B][Kmax] float32: sum_j max(0, p_i(j) - q_i(j)), which is
 *               1 - alpha_i, the rejection probability of position i.
 *   final_row   [B] int32: the row the final token was drawn from (= n_b).
 */
typedef struct {
    float* p_x;
    float* q_x;
    float* resid_mass;
    int32_t* final_row;
} sv_diag;

/*
 * Per-call counters (device memory, accumulated: zero them before the first
 * call they should cover).  Only the positions the method walks count: the
 * tested positions up to and including the first rejection.
 *   sequences   sequences with valid outputs (n_b >= 0)
 *   invalid     sequences whose device data was unusable (n_b = -1)
 *   tested      draft positions tested (accept tests taken)
 *   accepted    of these, the accepted ones
 *   committed   tokens committed: sum over valid sequences of n_b + 1
 *   near_ties   sampling accept tests whose uniform lies within 1e-6 of its
 *               threshold p/q (the decisions a change of summation order
 *               could flip)
 *   draw_near_ties  final draws (sampling sequences with valid outputs)
 *               whose point u lies within 1e-6 of a bound of the drawn
 *               token's interval [C_{j-1}, C_j) of the normalised CDF
 * The acceptance rate is accepted / tested; tokens per round is
 * committed / sequences.  (Before ABI version 4 the struct ended at
 * near_ties.)
 */
typedef struct {
    unsigned long long sequences;
    unsigned long long invalid;
    unsigned long long tested;
    unsigned long long accepted;
    unsigned long long committed;
    unsigned long long near_ties;
    unsigned long long draw_near_ties;
} sv_stats;

/*
 * Options for spec_verify_ex.  Zero-initialise for defaults.
 *   diag            diagnostics (requesting any forces verify_all).
 *   verify_all      1: sweep every row, including those after the first
 *                   rejection (the results are identical; only the work and
 *                   the diagnostics differ).  0: rows a known earlier
 *                   rejection makes irrelevant are skipped.
 *   chunks_per_cta  0: automatic.  Otherwise the number of vocabulary chunks
 *                   each CTA of a row's cluster holds (tuning: sets the
 *                   cluster size, at most 16; SV_ERR_UNSUPPORTED when the
 *                   row's slice then does not fit in shared memory).
 *   chunks_per_warp 0: automatic.  Otherwise how many of the CTA's chunks
 *                   each warp holds (tuning: sets the warps per CTA, at most
 *                   8 and at most 32 / cluster size).
 *   stats           device sv_stats to accumulate into, or NULL.
 *   kv_len          device [B] int32, or NULL: the caller's KV-cache lengths,
 *                   updated in place to kv_len[b] + 1 + n_b for every sequence
 *                   with valid outputs (unchanged when n_b = -1), so that no
 *                   host round trip is needed to commit the accepted tokens.
 *   packed_logits   0: the padded layouts above.  1: the logits of ragged
 *                   batches packed by K: target_logits [sum_b (K[b]+1)][V]
 *                   with sequence b's rows from row sum_{c<b} (K[c]+1), and
 *                   draft_logits [sum_b K[b]][V] with sequence b's rows from
 *                   row sum_{c<b} K[c].  Tokens, uniforms and outputs keep
 *                   their padded layouts.
 *   expire_copy_waits  testing only; 0 in normal use.  1: every bounded wait
 *                   for a row's copy into shared memory gives up before its
 *                   first poll, as a wait that ran out would.  This exercises
 *                   the timeout path: the rows of the affected sequences are
 *                   poisoned (their outputs -1), the workspace error word is
 *                   set (sv_workspace_errors returns SV_ERR_TIMEOUT), and the
 *                   copies already issued still land and are waited for, with
 *                   the normal bound, before the kernel exits.  Nothing faults
 *                   or hangs; the next call on the workspace is unaffected.
 *   temperature_host  host [B] float32, or NULL: a host copy of the device
 *                   `temperature` array, read during the call only.  It lets
 *                   the launch give the greedy sequences (T = 0, which read no
 *                   draft rows) to clusters split in two independent halves,
 *                   two greedy rows in the shared memory a sampling row
 *                   takes, while the other clusters take the sampling
 *                   sequences first.  The outputs are the same as without it.
 *                   Used by plain calls (no diagnostics, verify_all or tuning)
 *                   of the cluster kernel (V > 1024, 16-byte aligned rows)
 *                   with enough sequences of both kinds; ignored otherwise.
 *                   It must match the device array: a sequence it calls
 *                   greedy whose device temperature is not 0 (and K > 0, so
 *                   that it has draft rows to read) may get outputs -1 and
 *                   set bit 1 of the workspace error word
 *                   (sv_workspace_errors returns SV_ERR_INVALID_ARG).  A call
 *                   captured into a CUDA graph keeps the split it was
 *                   captured with: its replays need the same sequences
 *                   greedy.
 * Tuning options change only the fp32 summation grouping: results agree
 * with the automatic geometry except within the rounding of those sums.
 */
typedef struct {
    sv_diag diag;
    int32_t verify_all;
    int32_t chunks_per_cta;
    int32_t chunks_per_warp;
    sv_stats* stats;
    int32_t* kv_len;
    int32_t packed_logits;
    int32_t expire_copy_waits;
    const float* temperature_host;   /* since ABI version 5 */
} sv_options;

/* Human-readable name of a status code (static storage). */
const char* sv_status_string(sv_status status);

/* SV_ABI_VERSION of the loaded library. */
int32_t sv_abi_version(void);

/* Largest vocabulary size spec_verify accepts for dtype (0 for a bad dtype). */
int32_t sv_max_vocab(sv_dtype dtype);

/*
 * Launch geometry a call of this shape would use on the current device
 * (diagnostic; queries the device, queues no work).  out8 receives:
 *   [0] cluster size C (CTAs per row), [1] warps per CTA,
 *   [2] vocabulary chunks per warp, [3] clusters in the persistent grid,
 *   [4] threads per CTA, [5] dynamic shared memory per CTA (bytes),
 *   [6] warps whose range holds chunks, [7] vocabulary chunks per row.
 * Zero tuning arguments select the automatic choice (as in sv_options).
 */
sv_status sv_geometry(int32_t B, int32_t Kmax, int32_t V, sv_dtype dtype, int32_t chunks_per_cta,
                      int32_t chunks_per_warp, int32_t* out8);

/*
 * CUDA graphs.  spec_verify, spec_verify_ws, spec_verify_ex and spec_sample
 * may be called on a stream that is being captured, once an ordinary
 * (uncaptured) call of the same shape has run on the device: that call
 * reserves the pinned header a graph keeps (allocation is not allowed during
 * a capture) and records the launch geometry.  The graph holds the K and the
 * claim order of the captured call; at every replay it reads the logits,
 * tokens, uniforms and temperatures then in the captured buffers.  A capture
 * with no reserved header of its size returns SV_ERR_UNSUPPORTED, as do
 * spec_verify_host and spec_verify_noalloc on a capturing stream.
 */

/*
 * Bytes of device workspace spec_verify_ws / spec_verify_ex need for this
 * shape (0 on invalid arguments).  The workspace holds the error word, the
 * claim counter and a header-ready count, reset by every call on its stream.
 * The rest of the per-call header (K, the order in which sequences are
 * claimed, the packed row starts) is read by the kernel from a pinned,
 * device-mapped host buffer of the library's, which the kernel first copies
 * into the workspace when the batch has more sequences than the grid has
 * clusters; where pinned memory is unavailable or the caller's own host
 * staging is used (spec_verify_noalloc) it is uploaded into the workspace.
 * The buffer needs no clearing.
 */
size_t sv_workspace_size(int32_t B, int32_t Kmax, int32_t V, sv_dtype dtype);

/*
 * spec_verify -- verify B sequences (the entry point the pages' loop maps to).
 *   target_logits     device, [B][Kmax+1][V], dtype.
 *   draft_logits      device, [B][Kmax][V], dtype; may be NULL when every
 *                     temperature is 0 (a sampling sequence then yields -1).
 *   dtype             SV_DTYPE_F32 or SV_DTYPE_BF16 (both logit arrays).
 *   draft_tokens      device, [B][Kmax] int32; may be NULL iff Kmax == 0.
 *   uniforms          device, [B][Kmax+1] float32.
 *   temperature       device, [B] float32 (0 = greedy).
 *   B                 number of sequences, >= 0 (0 is a no-op).
 *   K                 HOST, [B] int32, 0 <= K[b] <= SV_K_MAX.
 *   V                 vocabulary size shared by target and draft, 1..sv_max_vocab.
 *   out_tokens        device, [B][Kmax+1] int32 (written).
 *   out_num_accepted  device, [B] int32 (written).
 *   stream            CUDA stream; all work is queued on it.
 * Scratch comes from the stream-ordered allocator (cudaMallocAsync) and is
 * released on the same stream.
 */
sv_status spec_verify(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                      const int32_t* draft_tokens, const float* uniforms,
                      const float* temperature, int32_t B, const int32_t* K, int32_t V,
                      int32_t* out_tokens, int32_t* out_num_accepted, cudaStream_t stream);

/* Size of the fixed scratch array spec_verify_noalloc works in (16 MiB). */
#define SV_STATIC_SCRATCH_BYTES (16u << 20)

/*
 * spec_verify_noalloc -- as spec_verify, for callers that cannot allocate
 * device memory at call time: a serving loop that has handed all free device
 * memory to its KV-cache pool (a cudaMalloc would fail there), or a caller
 * with no allocator of its own (plain C, no PyTorch) that must not pay an
 * allocation on every verification step.  The pages define no counterpart of
 * this entry point; it is the same verification as spec_verify_ws.
 *
 * Scratch: a fixed array of SV_STATIC_SCRATCH_BYTES in this library's own
 * device module (one per device), instead of a workspace argument.  Shapes
 * whose sv_workspace_size(B, Kmax, V, dtype) exceeds SV_STATIC_SCRATCH_BYTES
 * return SV_ERR_NO_MEMORY before any work is queued.  Nothing in the array
 * needs to start at zero: each call uploads the header it uses (error word,
 * claim counter, K and the claim order) before its kernel runs.  The per-call
 * header is assembled in a static host array.
 *
 * Set-up: the first call on a device resolves the array's address on that
 * device (cudaGetSymbolAddress, with the device current) and sets kernel
 * attributes; make that first call before any stream capture.  The first call
 * with a new shape also records its launch geometry in a small host cache.
 * No call allocates device memory (no cudaMalloc, cudaMallocAsync or
 * cudaFree).
 *
 * Calls share the one array per device and the one host header array:
 * overlapping calls (other streams, other host threads) race and give
 * undefined results.  Order them on one stream, from one host thread.
 * sv_workspace_errors does not apply (there is no workspace handle).
 */
sv_status spec_verify_noalloc(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                              const int32_t* draft_tokens, const float* uniforms,
                              const float* temperature, int32_t B, const int32_t* K, int32_t V,
                              int32_t* out_tokens, int32_t* out_num_accepted, cudaStream_t stream);

/*
 * spec_verify_ws -- as spec_verify, with a caller-provided device workspace of
 * at least sv_workspace_size(B, Kmax, V, dtype) bytes, 256-byte aligned.
 * Calls that share one workspace must be ordered on one stream.
 */
sv_status spec_verify_ws(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                         const int32_t* draft_tokens, const float* uniforms,
                         const float* temperature, int32_t B, const int32_t* K, int32_t V,
                         int32_t* out_tokens, int32_t* out_num_accepted,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * spec_verify_ex -- as spec_verify_ws plus options (may be NULL) and the
 * per-position diagnostics.
 */
sv_status spec_verify_ex(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                         const int32_t* draft_tokens, const float* uniforms,
                         const float* temperature, int32_t B, const int32_t* K, int32_t V,
                         int32_t* out_tokens, int32_t* out_num_accepted,
                         const sv_options* options, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/*
 * Device-side error flags recorded in a workspace by the last call that used
 * it (bit 0: a bounded shared-memory copy wait gave up; bit 1: a sequence
 * sv_options.temperature_host called greedy had a nonzero device
 * temperature).  Copies the word to *flags, clears it, and synchronises
 * `stream`.  Returns SV_ERR_TIMEOUT when bit 0 was set, else
 * SV_ERR_INVALID_ARG when bit 1 was, SV_OK otherwise.
 */
sv_status sv_workspace_errors(void* workspace, uint32_t* flags, cudaStream_t stream);

/*
 * spec_sample -- draw one token per row from softmax(logits[b] / T_b) by the
 * inverse CDF at uniforms[b] (the draft model's own sampling step, with the
 * machinery of the final draw: a K = 0 verification of every row).  A batch
 * of at least twice as many rows as the launch has clusters runs on split
 * clusters, two rows in the shared memory one verification row takes (as
 * does any all-K = 0 call of spec_verify_ws / spec_verify_ex).
 *   logits        device, [B][V], dtype.
 *   uniforms      device, [B] float32 in [0, 1).
 *   temperature   device, [B] float32 (0 = argmax, lowest index on ties).
 *   out_tokens    device, [B] int32 (written; -1 for a row with unusable data).
 *   workspace     device, at least sv_sample_workspace_size(B, V, dtype) bytes,
 *                 256-byte aligned.
 * Errors as spec_verify_ws.
 */
sv_status spec_sample(const void* logits, sv_dtype dtype, const float* uniforms,
                      const float* temperature, int32_t B, int32_t V, int32_t* out_tokens,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Bytes of device workspace spec_sample needs (0 on invalid arguments). */
size_t sv_sample_workspace_size(int32_t B, int32_t V, sv_dtype dtype);

/*
 * Bytes of device staging spec_verify_host needs (inputs, outputs and the
 * workspace), 0 on invalid arguments.
 */
size_t sv_host_staging_size(int32_t B, int32_t Kmax, int32_t V, sv_dtype dtype);

/*
 * spec_verify_host -- the same operation on HOST arrays (same layouts as
 * above).  `device_staging` is >= sv_host_staging_size bytes, 256-byte
 * aligned.  Logits in page-locked host memory that is mapped into the
 * device's address space (cudaHostAlloc / cudaHostRegister memory on a
 * system with unified addressing) are read in place by the kernel: only the
 * rows the method reaches cross the host link (on a Grace-Blackwell node,
 * NVLink-C2C).  Other logits (pageable memory) are first copied into the
 * staging.  Tokens, uniforms and temperatures are copied into the staging;
 * out_tokens / out_num_accepted are copied back to the host arrays, and
 * `stream` is synchronised before returning (the host arrays must not change
 * while the call runs).
 */
sv_status spec_verify_host(const void* h_target_logits, const void* h_draft_logits,
                           sv_dtype dtype, const int32_t* h_draft_tokens,
                           const float* h_uniforms, const float* h_temperature, int32_t B,
                           const int32_t* K, int32_t V, int32_t* h_out_tokens,
                           int32_t* h_out_num_accepted, void* device_staging,
                           size_t staging_bytes, cudaStream_t stream);

/*
 * spec_verify_tree -- token-tree verification: the accept rule of
 * spec_verify applied at every node of a tree of proposals (a tree of one
 * child per node is spec_verify).  Pages: tech-tldr.com "投機的デコーディング
 * とドラフトモデル", section 受理判定の数理 (the accept rule and the
 * distribution drawn from after a rejection); issoh.co.jp, section 受理・棄却
 * の規則と出力分布が変わらない理由 (losslessness).
 *
 * Per sequence b: nodes 0 .. n_nodes[b] - 1 (1 <= n_nodes[b] <= Nmax <= 32),
 * node 0 the root; parent[b][n] < n for n >= 1.  The candidates at node v are
 * its children (the nodes whose parent is v) in increasing index.  Row n of
 * the target / draft logits ([B][Nmax][V], device, dtype) is the target's /
 * draft's distribution after node n (the draft row is the one n's children
 * were drawn from; it is read only at sampling nodes with children, and
 * draft_logits may be NULL if every sequence is greedy).  tokens[b][n] is
 * node n's token; uniforms[b][n] (n >= 1) tests node n and uniforms[b][0] is
 * the final draw; temperature[b] as in spec_verify; all device, [B][Nmax] /
 * [B]; n_nodes is device memory too.
 *
 * Walk from the root: at node v, with R = p = softmax(target_v / T), child c
 * (token x) is kept iff u_c < min(1, R(x) / q(x)), q = softmax(draft_v / T);
 * a kept child is the next node; after a rejection R becomes
 * normalize(max(0, R - q)) (unchanged if that has no mass) and the next
 * child is tested.  With no child kept the token is drawn from R by inverse
 * CDF with uniforms[b][0] (at a leaf R = p, the bonus token).  At T = 0 the
 * child equal to the target argmax is kept, else the token is the argmax.
 *
 * Outputs (device, [B][Nmax]): out_path[b][0 .. len-1] the kept nodes,
 * out_tokens[b][0 .. len-1] their tokens and out_tokens[b][len] the drawn
 * token, -1 after; out_len[b] = len, or -1 (and -1 everywhere) when the
 * walk meets unusable input (a malformed tree, temperature, token, uniform
 * or row).  workspace: >= sv_tree_workspace_size() bytes, 256-byte aligned,
 * holds the error word (sv_workspace_errors).  Asynchronous on `stream`.
 */
size_t sv_tree_workspace_size(void);
sv_status spec_verify_tree(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                           const int32_t* tokens, const int32_t* parent, const float* uniforms,
                           const float* temperature, int32_t B, int32_t Nmax, const int32_t* n_nodes,
                           int32_t V, int32_t* out_tokens, int32_t* out_path, int32_t* out_len,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
