/*
 * ulysses.h -- C ABI of the GB300 (sm_103a) DeepSpeed-Ulysses attention block.
 *
 * The operations are those of one Transformer layer's attention under Ulysses sequence
 * parallelism, as described in "DeepSpeed Ulysses: System Optimizations for Enabling
 * Training of Extreme Long Sequence Transformer Models" (paper summary, section 3.2
 * "Big-Picture Architecture" and section 3.4.1 "Data Partitioning and Layout
 * Transformation"; pinyu.ai page "Ulysses Sequence Parallelism: A Temporary Change of
 * Layout", section "One attention block, end to end"):
 *   1. Q, K, V arrive as P token shards [B, L/P, H, d_h];
 *   2. a sequence-to-head all-to-all gives each of P head groups the full sequence for
 *      H/P heads, [B, L, H/P, d_h];
 *   3. exact attention O_h = softmax(Q_h K_h^T / sqrt(d_h) + mask) V_h runs per head;
 *   4. a head-to-sequence all-to-all returns O to [B, L/P, H, d_h].
 * The P "ranks" are P shards of one allocation in one GPU's memory, so each all-to-all is
 * an on-device permutation.
 *
 * Notation: Lp = L / P, Hp = H / P, global token s = r * Lp + t for shard r, local token
 * t; head group g owns heads h = g * Hp + j.
 *
 * Layouts (all contiguous, row-major, element = bf16 unless stated):
 *   ULYSSES_LAYOUT_TOKEN_SHARDED  [P][B][Lp][H][d_h]   (shard r = one rank's tensor)
 *   ULYSSES_LAYOUT_HEAD_SHARDED   [P][B][L][Hp][d_h]   (group g = one rank's tensor)
 *   log-sum-exp (fp32, natural log of the scaled scores)  [P][B][Hp][L]
 * Key/value tensors (K, V, dK, dV) have H_kv heads in place of H: token-sharded
 * [P][B][Lp][H_kv][d_h], head-sharded [P][B][L][Hkvp][d_h] with Hkvp = H_kv / P, or 1 when
 * P > H_kv (group g then holds a copy of key/value head g / (P / H_kv)).
 *
 * Conventions for every call below:
 *   - Ownership: the caller allocates and owns every buffer. The library allocates no
 *     device memory. Its state is a per-process error word on each device and, for each host
 *     thread, a cache of tensor maps and the USP forward's side streams; ulysses_shutdown()
 *     releases the calling thread's part.
 *   - Pointers are device pointers unless stated. `stream` is a cudaStream_t passed as
 *     void* (NULL = the legacy default stream). Calls enqueue work and return without
 *     synchronising; a launch failure returns ULYSSES_ERR_CUDA.
 *   - Arguments are validated before any launch: bad sizes or null pointers give
 *     ULYSSES_ERR_INVALID_ARG, buffers not 16-byte aligned give ULYSSES_ERR_MISALIGNED,
 *     valid but unimplemented cases give ULYSSES_ERR_UNSUPPORTED. Nothing is launched
 *     when a call fails.
 *   - Sizes with B == 0 or L == 0 are valid and launch nothing.
 *   - In-place operation is not supported; overlapping inputs and outputs are undefined
 *     (identical base pointers are rejected).
 *   - bf16 results are rounded to nearest-even from fp32. Relayouts move 16-bit patterns
 *     unchanged, NaN payloads included.
 *   - Every wait inside a kernel is bounded (about two seconds). A kernel that runs out
 *     of time records the fact in the device error word and returns early; read it with
 *     ulysses_get_device_status(). The word holds (kernel << 24) | (role << 16) | site of the
 *     first wait that gave up: kernel 1 forward, 2 backward, 3 self-test, 4 projection
 *     GEMM; role 1 loads, 2 MMA issue, 3 softmax, 4 dQ reduction, 5 epilogue, 6 self-test.
 */
#ifndef ULYSSES_H
#define ULYSSES_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ULYSSES_OK = 0,
    ULYSSES_ERR_INVALID_ARG = 1,
    ULYSSES_ERR_UNSUPPORTED = 2,
    ULYSSES_ERR_MISALIGNED = 3,
    ULYSSES_ERR_CUDA = 4,
    ULYSSES_ERR_DEVICE_TIMEOUT = 5
} ulysses_status_t;

typedef enum {
    ULYSSES_LAYOUT_TOKEN_SHARDED = 0,
    ULYSSES_LAYOUT_HEAD_SHARDED = 1
} ulysses_layout_t;

typedef enum {
    ULYSSES_MASK_NONE = 0,          /* bidirectional: every (query, key) pair          */
    ULYSSES_MASK_CAUSAL = 1,        /* key s' permitted for query s iff s' <= s         */
    ULYSSES_MASK_BLOCK_SPARSE = 2   /* whole tile x tile blocks from the lists below    */
} ulysses_mask_kind_t;

/* Shape of one attention block: batch B, sequence L (the paper's N), H query heads of width
 * d_h, P shards. Requires H % P == 0 and L % P == 0 (the head cut and the token cut must
 * be even; pinyu.ai page, "Head-count constraints").
 * H_kv: number of key/value heads (grouped-query attention; the pinyu.ai page's head-count
 * constraints and the paper summary's discussion of GQA/MQA). 0 means H (multi-head
 * attention). Query head h attends with key/value head h / (H / H_kv). Requires
 * H % H_kv == 0 and either H_kv % P == 0 (each head group receives H_kv / P whole
 * key/value heads) or P % H_kv == 0 (each head group receives one key/value head, replicated
 * on P / H_kv groups). */
typedef struct {
    int B, L, H, d_h, P;
    int H_kv;
} ulysses_shape_t;

/* Attention mask. For ULYSSES_MASK_BLOCK_SPARSE (a sparsity pattern applied locally after
 * the all-to-all, paper summary section 3.4.5 "Attention-Agnostic Design"): tile must be
 * 128; with n = ceil(L / 128) tiles,
 *   q_rowptr[n + 1], q_kcols[nnz]  -- CSR: key tiles of each query tile, ascending;
 *   k_colptr[n + 1], k_qrows[nnz]  -- CSC: query tiles of each key tile, ascending;
 * all int32 device arrays describing the same pattern (ulysses_bsmask_build_window_global
 * builds a consistent pair on the host). A permitted tile admits every pair inside it.
 * The same pattern applies to every batch entry and head. Lists that disagree with each
 * other give undefined results. Other kinds ignore these fields. */
typedef struct {
    int kind;
    int tile;
    const int32_t *q_rowptr;
    const int32_t *q_kcols;
    const int32_t *k_colptr;
    const int32_t *k_qrows;
    int nnz;
} ulysses_mask_t;

/* Sequence-to-head relayout (the first all-to-all; paper summary section 3.4.1, pinyu.ai
 * page "Use the other independent axis"):
 *   out[g][b][s][j][e] = in[s / Lp][b][s % Lp][g * Hp + j][e].
 * in: TOKEN_SHARDED bf16 (any 16-bit type), out: HEAD_SHARDED, both B*L*H*d_h elements.
 * Any d_h >= 1 is accepted; buffers need only 2-byte alignment. */
int ulysses_seq_to_head(ulysses_shape_t shape, const void *in, void *out, void *stream);

/* Head-to-sequence relayout (the second all-to-all, "After attention: the reverse
 * transformation"), the inverse permutation:
 *   out[r][b][t][h][e] = in[h / Hp][b][r * Lp + t][h % Hp][e]. */
int ulysses_head_to_seq(ulysses_shape_t shape, const void *in, void *out, void *stream);

/* Key/value sequence-to-head relayout, the first all-to-all applied to K or V with H_kv
 * heads (the seq->head relayout above with the receiver rule for grouped key/value heads):
 *   out[g][b][s][j][e] = in[s / Lp][b][s % Lp][src(g, j)][e],
 *   src(g, j) = g * Hkvp + j when H_kv % P == 0, else g / (P / H_kv) (replicated).
 * in: [P][B][Lp][H_kv][d_h], out: [P][B][L][Hkvp][d_h], 16-bit elements moved unchanged.
 * Only B, L, d_h, P and H_kv (H when H_kv is 0) are used: it needs L % P == 0 and
 * H_kv % P == 0 or P % H_kv == 0, but not H % P == 0. With H_kv == H it equals
 * ulysses_seq_to_head. */
int ulysses_kv_seq_to_head(ulysses_shape_t shape, const void *in, void *out, void *stream);

/* Adjoint of ulysses_kv_seq_to_head, for head-sharded key/value gradients: every key/value
 * head receives the sum over its copies,
 *   out[r][b][t][h][e] = sum over (g, j) with src(g, j) == h of in[g][b][r * Lp + t][j][e].
 * bf16 in and out; the sum is formed in fp32 in ascending g and rounded to nearest-even.
 * Without replication each head has one copy and this is the exact inverse permutation. */
int ulysses_kv_head_to_seq_sum(ulysses_shape_t shape, const void *in, void *out, void *stream);

/* One rank's side of the two all-to-alls when the P ranks are P processes (paper summary
 * section 3.4.2 "The All-to-All Communication Primitive"; aifetchly guide, "Explanation of the
 * Implementation", item 2): the collective itself (an NCCL all-to-all) belongs to the caller,
 * and these calls lay out its buffers. shape gives the whole problem: B, L (all ranks'
 * tokens), H (the tensor's own head count: H_kv for keys and values; shape.H_kv is ignored),
 * d_h and P; it needs H % P == 0 and L % P == 0.
 *   pack:   in  = this rank's token shard [B][L/P][H][d_h];
 *           out = [P][B][L/P][H/P][d_h], chunk g (heads [g H/P, (g+1) H/P)) to be sent to rank g:
 *           out[g][b][t][j][e] = in[b][t][g * H/P + j][e].
 *   unpack: the inverse: in = the P chunks received, chunk g from the rank holding head
 *           group g; out = [B][L/P][H][d_h].
 * With B = 1 the chunks an all-to-all delivers to rank g, concatenated in sender order, are
 * the head-sharded [L][H/P][d_h] of head group g. 16-bit elements moved unchanged; in and
 * out must not overlap; 2-byte alignment (16-byte for the vectorised path). */
int ulysses_a2a_pack(ulysses_shape_t shape, const void *in, void *out, void *stream);
int ulysses_a2a_unpack(ulysses_shape_t shape, const void *in, void *out, void *stream);

/* Attention forward for every head group (paper summary section 3.4.1 "The challenge at
 * the attention boundary", pinyu.ai page "The layout that saves memory breaks at
 * attention"):  S = scale * Q K^T + mask,  O = softmax(S) V,  lse = ln sum exp(S).
 * q, k, v, o: bf16 in io_layout (k, v with H_kv heads); with TOKEN_SHARDED the two relayouts
 * are fused into the kernel's loads and stores, so o comes back token-sharded.
 * lse: fp32 [P][B][Hp][L].
 * softmax_scale <= 0 selects 1/sqrt(d_h). A row with no permitted key gets O = 0 and
 * lse = -inf.
 * Supported: d_h in {64, 128}. TOKEN_SHARDED additionally needs Lp % 8 == 0. Any L >= 1
 * otherwise (a last partial tile is masked). Pointers 16-byte aligned. */
int ulysses_attn_fwd(ulysses_shape_t shape, const ulysses_mask_t *mask, float softmax_scale,
                     int io_layout, const void *q, const void *k, const void *v,
                     void *o, float *lse, void *stream);

/* Bytes of device workspace ulysses_attn_bwd needs for this shape (an fp32 dQ
 * accumulator and the per-row Delta = rowsum(dO * O)). */
size_t ulysses_attn_bwd_workspace_size(ulysses_shape_t shape);

/* Attention backward (the analytic gradient of the forward above; the pages do not write
 * it out). With P = exp(S - lse) on permitted pairs, Delta = rowsum(dO * O):
 *   dV = P^T dO,  dS = P * (dO V^T - Delta),  dQ = scale dS K,  dK = scale dS^T Q.
 * q, k, v, o, dO, dq, dk, dv: bf16 in io_layout (TOKEN_SHARDED fuses the relayout of dO
 * in and of dq, dk, dv out; k, v, dk, dv with H_kv heads); lse as written by
 * ulysses_attn_fwd. With grouped key/value heads, dk and dv hold the sum over the query heads
 * of each group; with HEAD_SHARDED and replicated key/value heads (P > H_kv), each group's
 * copy receives its own query heads' part, and ulysses_kv_head_to_seq_sum adds the copies. workspace: at least
 * ulysses_attn_bwd_workspace_size(shape) bytes, 256-byte aligned, caller-owned, contents
 * need not be initialised. dq accumulates in fp32 with atomic adds, so its bits may vary
 * from run to run by fp32 rounding; dk and dv are deterministic. */
int ulysses_attn_bwd(ulysses_shape_t shape, const ulysses_mask_t *mask, float softmax_scale,
                     int io_layout, const void *q, const void *k, const void *v,
                     const void *o, const float *lse, const void *dO,
                     void *dq, void *dk, void *dv,
                     void *workspace, size_t workspace_bytes, void *stream);

/* Size of the fixed device array behind ulysses_attn_bwd_noalloc (96 MiB). */
#define ULYSSES_BWD_NOALLOC_SCRATCH_BYTES (96u * 1024u * 1024u)

/* ulysses_attn_bwd without a workspace argument, for callers that cannot allocate device
 * memory (for instance code whose device memory is owned entirely by a host framework's
 * pool, or a runtime that may not call cudaMalloc after start-up). This entry point has no
 * counterpart on the pages; it only changes where the workspace lives. It allocates
 * nothing: the workspace is a file-scope device array of ULYSSES_BWD_NOALLOC_SCRATCH_BYTES
 * that every GPU loading the library holds until the process exits.
 *   - Arguments and results are those of ulysses_attn_bwd.
 *   - Returns ULYSSES_ERR_UNSUPPORTED, launching nothing, when
 *     ulysses_attn_bwd_workspace_size(shape) exceeds ULYSSES_BWD_NOALLOC_SCRATCH_BYTES
 *     (for example B=1, L=8192, H=16, d_h=128 fits; B=1, L=32768, H=32, d_h=128 does not).
 *     This size check comes first: such a shape returns ULYSSES_ERR_UNSUPPORTED even when
 *     another argument (mask, layout, d_h, a pointer) is also invalid. Shapes that fit are
 *     then validated exactly as ulysses_attn_bwd validates them.
 *   - The first call on a device looks up the array's device address with that device
 *     current; make that first call before any stream capture.
 *   - Every call on a device shares the one array, which keeps the contents of the last
 *     call (the kernels re-zero what must start at zero). Calls whose work overlaps on the
 *     GPU, from different streams or threads, race on it and give undefined results. */
int ulysses_attn_bwd_noalloc(ulysses_shape_t shape, const ulysses_mask_t *mask, float softmax_scale,
                             int io_layout, const void *q, const void *k, const void *v,
                             const void *o, const float *lse, const void *dO,
                             void *dq, void *dk, void *dv, void *stream);

/* The projections on either side of the attention block (paper summary section 3.2
 * "Big-Picture Architecture" and section 3.4.1 "Before attention"; pinyu.ai page "One
 * attention block, end to end"): every rank projects its own token shard, so over the
 * token-sharded layout both are matrix products over the M = B * L token rows
 * [P][B][Lp], y = x W^T, bf16 in and out with fp32 accumulation.
 *
 * QKV projection: x [P][B][Lp][hidden]; w_qkv [(H + 2 H_kv) d_h][hidden], rows ordered
 * Q heads, K heads, V heads. Writes q [P][B][Lp][H][d_h], k and v [P][B][Lp][H_kv][d_h],
 * the token-sharded layout ulysses_attn_fwd reads (no relayout in between).
 * Requires hidden, H d_h and H_kv d_h multiples of 32 (else ULYSSES_ERR_UNSUPPORTED);
 * pointers 16-byte aligned. */
int ulysses_qkv_proj(ulysses_shape_t shape, int hidden, const void *x, const void *w_qkv, void *q, void *k,
                     void *v, void *stream);

/* Output projection: o [P][B][Lp][H][d_h] (as ulysses_attn_fwd returns it, token-sharded);
 * w_o [hidden][H d_h]; writes y [P][B][Lp][hidden]. Same requirements. */
int ulysses_out_proj(ulysses_shape_t shape, int hidden, const void *o, const void *w_o, void *y, void *stream);

/* Ulysses-ring hybrid (the aifetchly page's step 5, "USP"; Ring Attention in the reading notes,
 * section 5.2), which lifts the P <= H limit of the head cut: P = P_u * P_ring. The sequence is
 * cut into P_ring ring blocks of L / P_ring tokens, i.e. P_u = P / P_ring consecutive token
 * shards each. Inside a block the Ulysses relayout spreads the heads over P_u head groups (so
 * P_u, not P, must divide H); across blocks each query block meets every key/value block, and
 * the block results are merged with the online-softmax rule (m = max lse_j, lse = m +
 * ln sum exp(lse_j - m), O = sum exp(lse_j - lse) O_j).
 * q, k, v, o, dO, dq, dk, dv: TOKEN_SHARDED [P][B][Lp][H (or H_kv)][d_h] as for
 * ulysses_attn_fwd with P shards. lse: fp32, per ring block the layout of that block's
 * attention, [P_ring][P_u][B][H / P_u][L / P_ring]. Masks: causal (by global token position) or
 * none; block-sparse gives ULYSSES_ERR_UNSUPPORTED. P_ring <= 64 and P % P_ring == 0; every
 * ring block must be a valid ulysses_attn_fwd shape. workspace: at least
 * ulysses_usp_workspace_size(shape, P_ring) bytes, 256-byte aligned (0 for invalid shapes). The
 * forward merges each query block's pairs into an fp32 running (O, lse) and rounds O to bf16
 * once. With a causal mask it runs the first query block (a single pair) on a second stream
 * that the library keeps for each host thread and device. That stream waits for `stream` at
 * the start of the call, and `stream` waits for it at the end through an event, so the call
 * keeps stream order like every other call. The backward sums partial gradients over block
 * pairs in fp32, so all its outputs are deterministic up to the reduction order of each block
 * pair's dQ. */
size_t ulysses_usp_workspace_size(ulysses_shape_t shape, int P_ring);
int ulysses_usp_attn_fwd(ulysses_shape_t shape, int P_ring, const ulysses_mask_t *mask, float softmax_scale,
                         const void *q, const void *k, const void *v, void *o, float *lse, void *workspace,
                         size_t workspace_bytes, void *stream);
int ulysses_usp_attn_bwd(ulysses_shape_t shape, int P_ring, const ulysses_mask_t *mask, float softmax_scale,
                         const void *q, const void *k, const void *v, const void *o, const float *lse,
                         const void *dO, void *dq, void *dk, void *dv, void *workspace, size_t workspace_bytes,
                         void *stream);

/* Host helper: the block-sparse pattern "sliding window plus strided global key tiles".
 * Query tile qt gets key tiles max(0, qt - window_before) .. min(n - 1, qt + window_after)
 * and every kt with kt % global_stride == 0 (global_stride <= 0: none), n = ceil(L/tile).
 * Writes host arrays rowptr[n + 1], kcols[cap], colptr[n + 1], qrows[cap]; *nnz holds the
 * capacity on entry and the number of active tiles on return. Returns INVALID_ARG if the
 * capacity is too small (*nnz then holds the size needed) or arguments are bad. */
int ulysses_bsmask_build_window_global(int L, int tile, int window_before, int window_after,
                                       int global_stride, int32_t *rowptr, int32_t *kcols,
                                       int32_t *colptr, int32_t *qrows, int *nnz);

/* Health check of the bounded waits: enqueues one small kernel whose two waiting warps wait
 * on an mbarrier that nothing ever arrives on. They give up after the same limit as the
 * attention kernels (about two seconds), record ULYSSES_ERR_DEVICE_TIMEOUT in the device error
 * word and return, leaving the context usable. The next ulysses_get_device_status then
 * reports ULYSSES_ERR_DEVICE_TIMEOUT with detail (3 << 24) | (6 << 16) | site, site 1 or 2
 * (whichever warp ran out first). Returns ULYSSES_ERR_CUDA if the launch fails. */
int ulysses_selftest_timeout(void *stream);

/* Synchronises `stream`, then reads and clears the current device's error word.
 * Returns ULYSSES_OK, ULYSSES_ERR_DEVICE_TIMEOUT (a bounded wait ran out), or
 * ULYSSES_ERR_CUDA. When detail is not NULL it receives the raw word (kernel, role and
 * wait site of the first failure). */
int ulysses_get_device_status(void *stream, uint32_t *detail);

/* Human-readable name of a status code (static storage). */
const char *ulysses_status_string(int status);

/* Releases what the library keeps for the calling host thread: the side stream and its two
 * events on each device (made by ulysses_usp_attn_fwd), after waiting for their work, and the
 * thread's cache of tensor maps. Other threads' state is untouched, and the library allocates
 * no device memory of its own. Any call afterwards makes the state again as needed. Returns
 * ULYSSES_OK, or ULYSSES_ERR_CUDA if a wait or a device switch failed (the state is released
 * all the same). A thread that never used them makes no CUDA call here. */
int ulysses_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* ULYSSES_H */
