/*
 * spec_verify.h -- C ABI of the GB300 batched draft-verify step of
 * speculative decoding.
 *
 * What one call computes (the "Speculative Decoding and EAGLE-3" lesson,
 * factory.pai-world.com, sections "Invariant: Leviathan rejection
 * sampling", "Build it" steps 1-4 and "KV cache rollback"):
 *
 *   for each request b (independently):
 *     q_j = softmax(target_logits[b, j-1, :] / T_b)   j = 1..N+1  (verifier)
 *     p_j = softmax(draft_logits [b, j-1, :] / T_b)   j = 1..N    (drafter)
 *     walk j = 1..N left to right:
 *        accept d_j iff p_j(d_j) == 0 or u_j < min(1, q_j(d_j) / p_j(d_j))
 *        at the first rejection j*: emit one token sampled from the residual
 *        (q_j* - p_j*)_+ / ||(q_j* - p_j*)_+||_1 (from q_j* if that is all 0)
 *     if all N are accepted: emit a bonus token sampled from q_{N+1}
 *   T_b == 0 is the greedy argmax-match path: d_j is accepted iff it equals
 *   argmax target_logits[b, j-1, :] (lowest index on ties); the token after
 *   the accepted prefix is the argmax of the next target row; draft logits
 *   are not read.
 *
 * Random numbers: Philox4x32-10 (Salmon et al., "Parallel Random Numbers:
 * As Easy as 1, 2, 3", SC'11) with key = (seed low 32 bits, seed high 32
 * bits) and counter = (b, j, draw, 0); a word w gives the uniform
 * (w >> 8) * 2^-24.  Draw 0 is the accept test at 1-based position j and
 * uses word 0.  Draw 1 is the correction at j* or the bonus at j = N+1 and
 * uses all four words, u_1..u_4, in a grouped inverse CDF: the vocabulary
 * is cut into blocks of 8192 consecutive tokens (level 1), each block into
 * blocks of 256 (level 2), those into blocks of 16 (level 3) and those into
 * single tokens (level 4); level l picks, among the sub-blocks of the block
 * chosen so far, the smallest index whose running mass exceeds u_l times
 * their total mass (the last sub-block with mass if rounding leaves none).
 * The token is drawn exactly from the normalised residual (or q), since the
 * levels' conditional masses multiply to its probability.
 *
 * Layout: every tensor is dense row-major, caller-owned DEVICE memory
 * (cudaMalloc / torch CUDA tensors on the context's device).  Logits are
 * float32 or bfloat16 as fixed at init.  Rows whose byte offset is a
 * multiple of 16 (V * sizeof(elem) % 16 == 0 and 16-byte aligned bases)
 * take the vectorised path; any other V works through a scalar path.
 *
 * Calls are asynchronous on the stream given at init and never block the
 * host.  The library never aborts, traps or prints.  A single context must
 * not be used from two host threads at once; calls on one context are
 * ordered by its stream (the workspace is reused by the next call).
 */
#ifndef SPEC_VERIFY_H_
#define SPEC_VERIFY_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------ */
#define SV_OK          0  /* success                                          */
#define SV_EINVAL      1  /* host check: null pointer, size or dtype out of range */
#define SV_EBADTEMP    2  /* device check: a temperature is negative, NaN, inf
                             or a positive subnormal                           */
#define SV_EBADTOKEN   3  /* device check: a draft token outside [0, V)        */
#define SV_EBADLOGIT   4  /* device check: a row that is read holds NaN or +inf,
                             or all of its entries are -inf                    */
#define SV_ECUDA       5  /* a CUDA runtime call failed                        */
#define SV_ESCRATCH    6  /* spec_verify_noalloc: the problem's working memory
                             exceeds SV_NOALLOC_SCRATCH_BYTES                  */
#define SV_EBADTREE    7  /* device check (spec_verify_tree): a node's parent is
                             outside [0, node - 1]                             */
#define SV_EBADKV      8  /* device check (spec_verify_kv_commit): a sequence's
                             commit was refused                                */
#define SV_ETIMEOUT    9  /* a bounded device wait ran out and the kernel stopped
                             early (never expected; the context stays usable) */

/* Bits of the device error word (spec_verify_get_error).  A request that
 * fails a device check gets out_tokens = -1 everywhere, out_accept_len = -1
 * and out_kv_len = 0; the checks run in the order temperature, tokens,
 * (a bounded wait that ran out,) logits and only the first failing one is
 * recorded for the request. */
#define SV_ERRBIT_TEMP   1u
#define SV_ERRBIT_TOKEN  2u
#define SV_ERRBIT_LOGIT  4u
#define SV_ERRBIT_TREE   8u   /* spec_verify_tree only; checked after the
                                 temperature, before tokens and logits */
#define SV_ERRBIT_KV     16u  /* spec_verify_kv_commit only */
#define SV_ERRBIT_WAIT   32u  /* a bounded device wait ran out */

/* ---- logit element types ---------------------------------------------- */
typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;  /* int-sized in the C ABI */

/* Limits of one context. */
#define SV_MAX_N 255            /* drafts per request                       */
#define SV_MAX_V (1 << 26)      /* vocabulary size                          */

typedef struct spec_verify_ctx spec_verify_ctx;   /* opaque, library-owned */

/*
 * spec_verify_init -- create a context on the current CUDA device.
 *
 *   ctx          out: the new context (NULL on failure)
 *   max_B        1 .. 2^20 requests per call
 *   max_N        0 .. SV_MAX_N drafts per request
 *   max_V        1 .. SV_MAX_V vocabulary size
 *   dtype        SV_F32 or SV_BF16: element type of both logit tensors
 *   cuda_stream  cudaStream_t the calls are enqueued on (NULL = legacy
 *                default stream)
 *
 * Allocates the whole device workspace once (per-row partial statistics,
 * per-request walk results and sampling sums; a few MB at most) and zeroes
 * the parts that must start at zero.  The same context serves
 * spec_verify_tree with up to max_N draft nodes per tree.  Returns SV_OK, SV_EINVAL or SV_ECUDA.
 */
int spec_verify_init(spec_verify_ctx** ctx, int max_B, int max_N, int max_V,
                     sv_dtype dtype, void* cuda_stream);

/*
 * spec_verify -- one batched verify step.
 *
 *   B, N, V          0 <= B <= max_B, 0 <= N <= max_N, 1 <= V <= max_V
 *   target_logits    [B, N+1, V] dtype: rows j = 0..N give q_1..q_{N+1}
 *   draft_logits     [B, N, V] dtype: rows j = 0..N-1 give p_1..p_N
 *                    (may be NULL only when N == 0)
 *   draft_tokens     [B, N] int32, each in [0, V)
 *   temperature      [B] float32: 0 = greedy, else finite and >= 2^-126
 *   seed             64-bit Philox key
 *   out_tokens       [B, N+1] int32: the a_b accepted drafts, then the
 *                    correction or bonus token, then -1 padding
 *   out_accept_len   [B] int32: a_b in [0, N], drafts accepted
 *   out_kv_len       [B] int32: a_b + 1, KV entries of this verify window to
 *                    commit (the verified input token plus the accepted
 *                    drafts; the lesson's "KV cache rollback": the logical
 *                    length stops right after the correction token)
 *
 * B == 0 is a no-op.  Returns SV_OK, SV_EINVAL (nothing enqueued) or
 * SV_ECUDA.  Device-detected input errors do not change the return value:
 * they mark the request's outputs (see SV_ERRBIT_*) and are read with
 * spec_verify_get_error.  The sampling kernel starts on a request as soon
 * as that request's rows are reduced, by polling tags on the partial
 * statistics; the tag is a per-call sequence number the context keeps on
 * the host, so every call is enqueued by the host (a replay of one captured
 * call would reuse its number).  A poll that runs out (about a second, only
 * if the row kernel stalls) marks the request with SV_ERRBIT_WAIT.
 */
int spec_verify(spec_verify_ctx* ctx, int B, int N, int V,
                const void* target_logits, const void* draft_logits,
                const int32_t* draft_tokens, const float* temperature,
                uint64_t seed, int32_t* out_tokens, int32_t* out_accept_len,
                int32_t* out_kv_len);

/*
 * spec_verify_noalloc -- the same verify step as spec_verify, for callers
 * that may not allocate device memory while they run (for instance a
 * serving runtime that has handed all of HBM to its own KV-cache and
 * activation pools, or that cannot afford the device-wide synchronisation
 * of a cudaMalloc / cudaFree inside its decode loop).  The method itself
 * has no counterpart to this entry point: it exists only for that kind of
 * caller.
 *
 * No context: the call takes B, N, V, dtype (SV_F32 or SV_BF16) and the
 * stream directly; the tensors, seed and outputs are exactly those of
 * spec_verify and the results are identical to a spec_verify call with the
 * same inputs.  The library allocates nothing: the working memory comes
 * from one static device array of SV_NOALLOC_SCRATCH_BYTES bytes in the
 * library, and the call makes no cudaMalloc, cudaFree or other allocating
 * call.  The working memory is about
 *     B (2N+1) (16 ceil(V / C) + 8) + B (8 ceil(V / 8192) + 4 N + 4)  bytes,
 * C = 32768 elements for bfloat16 and 16384 for float32 logits (plus
 * 256-byte alignment of each part); problems that need more are refused
 * with SV_ESCRATCH before anything is enqueued.  B = 64 requests with
 * N = 7 drafts over V = 128256 bfloat16 logits need about 80 KB.
 *
 * Set-up: the first call on a device (with that device current) looks up
 * the array's device address with cudaGetSymbolAddress and caches it for
 * that device; make that first call before any stream capture starts.
 *
 * Sharing: all calls on a device use the same array.  Calls must be ordered
 * (one stream, or streams ordered by events): two calls whose kernels
 * overlap corrupt each other's results.  Each call clears its device error
 * word, its sampling counters and the tags of its partial statistics (one
 * memset) before its kernels run; device-detected input errors are reported in
 * the request's outputs only (out_tokens -1, out_accept_len -1,
 * out_kv_len 0; see SV_ERRBIT_*), since there is no context to read them
 * from.
 *
 * Returns SV_OK, SV_EINVAL (nothing enqueued), SV_ESCRATCH (nothing
 * enqueued) or SV_ECUDA.
 */
#define SV_NOALLOC_SCRATCH_BYTES (1u << 20)
int spec_verify_noalloc(int B, int N, int V, sv_dtype dtype,
                        const void* target_logits, const void* draft_logits,
                        const int32_t* draft_tokens, const float* temperature,
                        uint64_t seed, int32_t* out_tokens,
                        int32_t* out_accept_len, int32_t* out_kv_len,
                        void* cuda_stream);

/*
 * spec_verify_tree -- one batched verify step over a draft TREE instead of
 * a chain (the lesson's "Key terms" entry on EAGLE-2's dynamic draft tree,
 * its tree-mask remark in "KV cache rollback", and exercise 3's [2, 2, 2]
 * tree of eight candidate paths scored by one verifier pass).
 *
 * Layout per request: node 0 is the root (the last verified token), draft
 * nodes are 1..M in topological order.
 *   parents          [B, M] int32: parent of node i+1, in [0, i]
 *   draft_tokens     [B, M] int32: token of node i+1, in [0, V)
 *   target_logits    [B, M+1, V] dtype: row r = the verifier's next-token
 *                    logits after node r (the tree-masked forward pass)
 *   draft_logits     [B, M+1, V] dtype: row r = the drafter's logits from
 *                    which node r's children were drawn (read only in
 *                    SV_TREE_SAMPLED mode, and only rows of nodes that have
 *                    children); may be NULL in SV_TREE_TOPK mode
 *   temperature      [B] float32, seed: as for spec_verify
 *   mode             SV_TREE_SAMPLED: the children of a node are independent
 *                    draws from its draft row; SV_TREE_TOPK: they are fixed
 *                    candidates (e.g. the drafter's top-k), tested as draws
 *                    from a point mass on their own token
 * The walk starts at the root; the children of the current node are tried
 * in increasing node index (list siblings most probable first).  Child x is
 * accepted iff p(x) = 0 or u < min(1, r(x) / p(x)), r the node's current
 * distribution (q at first, after a rejection (r - p)_+ renormalised; in
 * TOPK mode p is the point mass, so r(x) decides and the residual drops x).
 * Accepting descends into the child; when every child is rejected a token
 * is drawn from the final r, and at a leaf a bonus token from its q.  Both
 * modes keep the verifier's law exactly.  Uniforms: the i-th child tried at
 * depth j uses Philox counter (b, j, i == 0 ? 0 : i + 1, 0); the token drawn
 * at depth j uses draw 1 and the grouped inverse CDF of spec_verify, so a
 * tree with one child per node gives exactly spec_verify's results.  T = 0
 * descends into the first child whose token is the node's target argmax.
 *
 * Outputs:
 *   out_tokens       [B, M+1] int32: the accepted path's tokens, then the
 *                    drawn token, then -1
 *   out_path         [B, M] int32: the accepted node indices (1..M), then -1
 *                    (the tree positions whose KV entries to keep)
 *   out_accept_len   [B] int32: path length a; out_kv_len [B]: a + 1
 * Limits: 0 <= M <= max_N of the context, B <= max_B, V <= max_V.  Device
 * errors mark the request (-1 / -1 / 0) and set SV_ERRBIT_* (temperature,
 * tree, token, logit, in that order).  Each rejection in SAMPLED mode costs
 * one extra pass over that node's two rows.  Returns SV_OK, SV_EINVAL
 * (nothing enqueued) or SV_ECUDA.  Two kernel launches per call.
 */
#define SV_TREE_SAMPLED 0
#define SV_TREE_TOPK    1
int spec_verify_tree(spec_verify_ctx* ctx, int B, int M, int V, int mode,
                     const void* target_logits, const void* draft_logits,
                     const int32_t* parents, const int32_t* draft_tokens,
                     const float* temperature, uint64_t seed,
                     int32_t* out_tokens, int32_t* out_path,
                     int32_t* out_accept_len, int32_t* out_kv_len);

/*
 * spec_verify_tree_lazy -- spec_verify_tree reading only the rows its walk
 * reaches (the lesson's "Invariant: Leviathan rejection sampling": a node's
 * children are tested against that node's rows alone, so the rows of nodes
 * the walk never reaches do not influence the result): when the walk
 * arrives at a node, the node's target row (and, in SV_TREE_SAMPLED mode,
 * its draft row if it has children) is reduced on the spot.  Same
 * arguments, layout, uniforms and outputs as spec_verify_tree; on valid
 * inputs the outputs are spec_verify_tree's bit for bit.  Errors: the
 * temperature, the topology and every token are checked first; a row is
 * checked only when the walk reads it, so a bad row of a node the walk
 * never reaches is not an error (spec_verify_tree checks every row).
 * Limit: rows of at most 32 spans of 64 KB (V <= 1048576 for SV_BF16,
 * 524288 for SV_F32), else SV_EINVAL.  One kernel launch per call, no
 * workspace traffic between kernels.
 */
int spec_verify_tree_lazy(spec_verify_ctx* ctx, int B, int M, int V, int mode,
                          const void* target_logits, const void* draft_logits,
                          const int32_t* parents, const int32_t* draft_tokens,
                          const float* temperature, uint64_t seed,
                          int32_t* out_tokens, int32_t* out_path,
                          int32_t* out_accept_len, int32_t* out_kv_len);

/*
 * spec_verify_lazy -- the same step as spec_verify (same arguments, same
 * outputs bit for bit on valid inputs), reading each request's rows only as
 * far as its walk goes: position j reads target row j-1 and draft row j-1
 * (target row j-1 alone at T = 0), the bonus / last greedy argmax reads
 * target row N, and rows after the first rejection are never read (the
 * lesson's "Invariant: Leviathan rejection sampling": the walk is left to
 * right and stops at the first rejection).  Fewer bytes when drafts are
 * rejected early; one dependent pass per position instead of one pass over
 * everything.  One kernel launch (a thread-block cluster per request).
 * Device checks: the temperature and every token first; a row is checked
 * when the walk reads it, so a bad row past the stop is not an error (the
 * one way its outputs can differ from spec_verify's).  Does not write the
 * statistics read by spec_verify_debug_stats.  Returns SV_OK, SV_EINVAL
 * (nothing enqueued) or SV_ECUDA.
 */
int spec_verify_lazy(spec_verify_ctx* ctx, int B, int N, int V,
                     const void* target_logits, const void* draft_logits,
                     const int32_t* draft_tokens, const float* temperature,
                     uint64_t seed, int32_t* out_tokens, int32_t* out_accept_len,
                     int32_t* out_kv_len);

/*
 * spec_verify_kv_commit -- commit the verifier's KV entries of the verify
 * window after spec_verify / spec_verify_tree (the lesson's "KV cache
 * rollback": the verify pass extends the cache by the window; entries past
 * the correction token are wrong; either write the window to a scratch
 * buffer and commit the accepted entries, or keep the physical cache and cut
 * the logical length back; exercise 4's two sequences).
 *
 *   mode         SV_KV_SCRATCH: the window is in `scratch` [L, B, W,
 *                entry_bytes]; kept window position i is copied to cache
 *                position seq_len[b] + i.
 *                SV_KV_INPLACE: the window was written into the cache at
 *                positions seq_len[b] + w; kept position i is moved from
 *                seq_len[b] + pos_i to seq_len[b] + i (a chain moves
 *                nothing); scratch may be NULL.
 *   cache        [L, B, S, entry_bytes] device bytes (all heads' K and V of
 *                one layer and position form one entry), 16-byte aligned;
 *                entry_bytes a multiple of 16
 *   seq_len      [B] int32, in/out: the logical length before the commit;
 *                it is advanced by kv_len[b]
 *   kv_len       [B] int32: out_kv_len of the verify step (<= 0: nothing
 *                kept, length unchanged)
 *   path         NULL for a chain (kept positions 0, 1, ..., kv_len - 1), or
 *                out_path of spec_verify_tree with row stride path_stride
 *                (kept positions 0, path[0], ..., path[kv_len - 2])
 * Entries past the new length are left as they are.  A sequence whose
 * commit would pass S, read outside the window, or keep positions that do
 * not rise is left unchanged and sets SV_ERRBIT_KV.  Enqueued on the
 * context's stream (two kernel launches); returns SV_OK, SV_EINVAL or
 * SV_ECUDA.  Uses only the context's stream and error word.
 */
#define SV_KV_SCRATCH 0
#define SV_KV_INPLACE 1
int spec_verify_kv_commit(spec_verify_ctx* ctx, int mode, int L, int B, int S, int W,
                          size_t entry_bytes, const void* scratch, void* cache,
                          int32_t* seq_len, const int32_t* kv_len,
                          const int32_t* path, int path_stride);

/*
 * spec_verify_fc_norm -- the drafter's input fusion of EAGLE-3 / EAGLE 3.1
 * (the EAGLE-3 page's "FC normalisation: the key change of EAGLE 3.1"):
 *     out = [norm(h_early); norm(h_mid); norm(h_late)] . W^T + bias
 * with the three target hidden states of an early, a middle and a late
 * layer.  norm: SV_NORM_NONE (EAGLE-3: plain concatenation), SV_NORM_LAYER
 * (LayerNorm: (h - mean) / sqrt(var + eps) * gamma + beta, the page's
 * formula) or SV_NORM_RMS (h / sqrt(mean(h^2) + eps) * gamma, the wording of
 * the EAGLE 3.1 news page); each segment has its own gamma / beta.
 *
 *   T, d, d_out   tokens, hidden width (a multiple of 64), output width
 *   h_early/mid/late  [T, d] bfloat16 device, 16-byte aligned
 *   gamma         [3, d] float32 (ignored for SV_NORM_NONE)
 *   beta          [3, d] float32 or NULL (LayerNorm only)
 *   weight        [d_out, 3 d] bfloat16, row-major, 16-byte aligned
 *   bias          [d_out] float32 or NULL
 *   out           [T, d_out] bfloat16 (caller-owned)
 *   xbuf          [T, 3 d] bfloat16 scratch (caller-owned, 16-byte aligned):
 *                 for LayerNorm / RMSNorm it receives the normalised,
 *                 concatenated input, which the GEMM then reads; with
 *                 SV_NORM_NONE the GEMM reads the hidden states themselves
 *                 and xbuf is left untouched
 * Statistics in float32; the normalised inputs are rounded to bfloat16 and
 * multiplied on the tensor cores (tcgen05, fp32 accumulation in tensor
 * memory); the output is rounded to bfloat16.  One kernel launch on the
 * context's stream for SV_NORM_NONE, two otherwise.  Returns SV_OK,
 * SV_EINVAL (nothing enqueued) or SV_ECUDA; a device wait that ran out is
 * reported by spec_verify_get_error as SV_ETIMEOUT.
 */
#define SV_NORM_NONE  0
#define SV_NORM_LAYER 1
#define SV_NORM_RMS   2
int spec_verify_fc_norm(spec_verify_ctx* ctx, int T, int d, int d_out, int norm, float eps,
                        const void* h_early, const void* h_mid, const void* h_late,
                        const float* gamma, const float* beta, const void* weight,
                        const float* bias, void* out, void* xbuf);

/*
 * spec_verify_get_error -- wait for the context's stream, then return the
 * first device-detected error since the last read (SV_EBADTEMP,
 * SV_EBADTREE, SV_EBADTOKEN, SV_EBADLOGIT, SV_EBADKV, SV_ETIMEOUT in that
 * priority) or SV_OK, and clear it.
 * bits (may be NULL) receives the OR of SV_ERRBIT_* flags.
 */
int spec_verify_get_error(spec_verify_ctx* ctx, uint32_t* bits);

/*
 * spec_verify_debug_stats -- copy the row statistics of the last
 * spec_verify call (same B, N; enqueued on the context's stream) into
 * caller-owned device buffers, for parity checks:
 *   accept_prob  [B, N] float32: min(1, q_j(d_j) / p_j(d_j)) (1 when
 *                p_j(d_j) == 0); NaN for greedy or failed requests
 *   log_z        [B, 2N+1] float32: per request, log sum_t exp(x_t / T) of
 *                target rows 0..N then draft rows 0..N-1 (natural log);
 *                NaN where the row was not normalised
 * Returns SV_OK, SV_EINVAL or SV_ECUDA.
 */
int spec_verify_debug_stats(spec_verify_ctx* ctx, int B, int N,
                            float* accept_prob, float* log_z);

/*
 * Kernel timing for benchmarks.  spec_verify_profile(ctx, every) with
 * every > 0 makes every every-th call of spec_verify, spec_verify_tree,
 * spec_verify_tree_lazy and spec_verify_lazy on the context (the first, then
 * each every-th after it;
 * 1 = all calls) record CUDA events around each kernel it launches on the
 * context's stream; every == 0 turns this off, and a negative value is
 * SV_EINVAL.  Events around kernels keep them from overlapping one another,
 * so recording a sample of the calls disturbs a timed loop less.
 * spec_verify_profile_read waits for the stream and returns, for the
 * recorded calls since the last read, the summed device time in
 * milliseconds of each of the SV_NUM_KERNELS kernel slots and the number of
 * recorded calls; it then clears the sums.  For spec_verify slot 0 is the
 * row-statistics kernel (every logit row streamed once, with the draft
 * tokens' logits) and slot 1 the walk and draw kernel; for spec_verify_tree
 * the same with the tree walk; spec_verify_lazy and spec_verify_tree_lazy
 * launch one kernel each (slot 0; slot 1 reads 0).
 */
#define SV_NUM_KERNELS 2
int spec_verify_profile(spec_verify_ctx* ctx, int every);
int spec_verify_profile_read(spec_verify_ctx* ctx, double* ms_per_kernel,
                             int* calls);

/* Number of kernel launches one spec_verify call with B > 0 makes (2). */
int spec_verify_launches_per_call(void);

/*
 * spec_verify_debug_philox -- test hook.  For i < n, writes the four
 * Philox4x32-10 output words of counter (ctr3[3i], ctr3[3i+1], ctr3[3i+2], 0)
 * under key (seed low 32 bits, seed high 32 bits) to out4[4i .. 4i+3],
 * using the same device function as the walk.  ctr3 and out4 are device
 * buffers; enqueued on cuda_stream.  Returns SV_OK, SV_EINVAL or SV_ECUDA.
 */
int spec_verify_debug_philox(uint64_t seed, const uint32_t* ctr3, uint32_t* out4, int n,
                             void* cuda_stream);

/*
 * spec_verify_debug_read_stream -- measurement hook: the achievable
 * streaming-read bandwidth of this GPU, reported beside the nominal and the
 * measured copy peaks as the row statistics' size-matched reference (what a
 * plain read of the same bytes achieves).  Reads the `bytes` bytes at buf
 * (device, 16-byte aligned, bytes a multiple of 16) once with 16-byte
 * non-allocating loads from a grid of 8 CTAs per SM (one kernel launch and
 * nothing else), and adds the sum of the buffer's 64-bit little-endian
 * words to the device word *out_sum, modulo 2^64, so no read can be
 * dropped (the caller clears *out_sum).  Enqueued on cuda_stream.  Returns
 * SV_OK, SV_EINVAL or SV_ECUDA.
 */
int spec_verify_debug_read_stream(const void* buf, size_t bytes, uint64_t* out_sum,
                                  void* cuda_stream);

/*
 * spec_verify_debug_skip_row_stats -- test hook for the bounded waits.  With
 * on != 0, the following spec_verify / spec_verify_tree calls on the context
 * launch their sampling (walk) kernel alone, without the row-statistics
 * kernel, so no partial statistics of those calls ever arrive: every poll
 * for them runs out (about a second), each request with a valid temperature
 * and valid tokens (and topology) is failed with SV_ERRBIT_WAIT, and
 * spec_verify_get_error returns SV_ETIMEOUT.  on == 0 restores normal calls;
 * the context stays usable throughout.  Host-side only: enqueues nothing.
 * Returns SV_OK or SV_EINVAL.
 */
int spec_verify_debug_skip_row_stats(spec_verify_ctx* ctx, int on);

/*
 * spec_verify_debug_late_cta -- test hook for a wait that runs out in one
 * sampler CTA of a request while the request's other CTAs finish.  With
 * cta >= 0, the following spec_verify calls on the context make the sampling
 * kernel's CTA number `cta` of every request (a request has one CTA per two
 * level-1 blocks of 8192 tokens for bfloat16 logits, one per block for
 * float32; CTA 0 also writes the walk's outputs) act as if its poll for the
 * row statistics ran out.  A sampled request with such a CTA is failed as a
 * whole (out_tokens -1, out_accept_len -1, out_kv_len 0, SV_ERRBIT_WAIT);
 * the counters the request's CTAs share carry the call's sequence number,
 * so a later call on the context is not disturbed.  cta == -1 restores
 * normal calls.  Host-side only: enqueues nothing.  Returns SV_OK or
 * SV_EINVAL.
 */
int spec_verify_debug_late_cta(spec_verify_ctx* ctx, int cta);

/*
 * spec_verify_debug_seek_calls -- test hook.  Sets the context's count of
 * spec_verify calls (the tag the next call's partial statistics carry is
 * calls + 1, wrapping past 2^32 - 1 to 1 after clearing every tag), so a
 * test can cross the wrap without 2^32 calls.  Host-side only: enqueues
 * nothing.  Returns SV_OK or SV_EINVAL.
 */
int spec_verify_debug_seek_calls(spec_verify_ctx* ctx, uint32_t calls);

/* Release the context and its workspace (waits for its stream first).
 * NULL is accepted.  Returns SV_OK or SV_ECUDA. */
int spec_verify_destroy(spec_verify_ctx* ctx);

/* Static, human-readable text for a return code. */
const char* spec_verify_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H_ */
