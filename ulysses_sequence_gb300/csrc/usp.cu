// Ulysses-ring hybrid ("USP" on the aifetchly page, step 5; Ring Attention in the reading
// notes, section 5.2): P = P_u x P_ring shards. The sequence is cut into P_ring contiguous ring
// blocks of L / P_ring tokens; each block is itself a token-sharded tensor of P_u = P / P_ring
// shards, inside which the Ulysses relayout spreads the H heads over P_u head groups (so only
// P_u, not P, must divide H). Across blocks, the key/value blocks are streamed past each query
// block and the per-block attention results are merged with the online-softmax rule:
//   m = max_j lse_j,  lse = m + ln sum_j exp(lse_j - m),  O = sum_j exp(lse_j - lse) O_j.
// The block-pair attentions are the library's own forward and backward on tensor slices: causal
// on the diagonal block pair and dense on every pair below it (on all pairs for a dense mask).
// The forward merges in the block-pair kernel's epilogue: a query block's first pair stores its
// normalised (O, lse) to an fp32 running pair, each later pair merges its own into it by the
// rule above, and the last pair writes O (rounded to bf16 once) and lse. The backward of a block
// pair uses the merged O and lse, so its probabilities are those of the whole row; its partial
// gradients are summed over block pairs in fp32 inside the block-pair backward (its dQ
// accumulator, and an fp32 store/add mode of its dK, dV epilogue).
#include "common.cuh"
#include "ulysses_internal.h"

namespace ulysses {

namespace {

struct UspGeom {
    ulysses_shape_t sub;    // one ring block: L / P_ring tokens, P / P_ring shards
    size_t q_elems, kv_elems, lse_elems;  // per ring block
    size_t acc_bytes, lse_bytes;          // the running O (fp32) and lse of one query block, 256-aligned
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

UspGeom usp_geom(const ulysses_shape_t& s, int P_ring) {
    UspGeom g{};
    g.sub = s;
    g.sub.L = s.L / P_ring;
    g.sub.P = s.P / P_ring;
    const size_t hkv = size_t(shape_hkv(s));
    g.q_elems = size_t(s.B) * g.sub.L * s.H * s.d_h;
    g.kv_elems = size_t(s.B) * g.sub.L * hkv * s.d_h;
    g.lse_elems = size_t(s.B) * s.H * g.sub.L;
    g.acc_bytes = align256(g.q_elems * 4);
    g.lse_bytes = align256(g.lse_elems * 4);
    return g;
}

// A second stream of this host thread on the current device, and two events, for the forward's
// query block that needs no running pair. They are made once per thread and device and never
// shared, so neither another thread's work nor another thread's stream capture can interleave
// with this thread's calls on them.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

constexpr int kSideDevs = 64;
thread_local SideStream t_side[kSideDevs];

bool side_stream(SideStream& out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kSideDevs) return false;
    SideStream& s = t_side[dev];
    if (!s.stream) {
        if (cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking) != cudaSuccess) {
            s.stream = nullptr;
            return false;
        }
        if (cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming) != cudaSuccess) {
            if (s.fork) cudaEventDestroy(s.fork);
            cudaStreamDestroy(s.stream);
            s = SideStream();
            return false;
        }
    }
    out = s;
    return true;
}

}  // namespace

bool release_side_streams() {
    int cur = -1;
    bool ok = true;
    for (int dev = 0; dev < kSideDevs; ++dev) {
        SideStream& s = t_side[dev];
        if (!s.stream) continue;
        if (cur < 0 && cudaGetDevice(&cur) != cudaSuccess) cur = 0;
        ok = cudaSetDevice(dev) == cudaSuccess && ok;
        ok = cudaStreamSynchronize(s.stream) == cudaSuccess && ok;
        cudaEventDestroy(s.fork);
        cudaEventDestroy(s.join);
        cudaStreamDestroy(s.stream);
        s = SideStream();
    }
    if (cur >= 0) ok = cudaSetDevice(cur) == cudaSuccess && ok;
    return ok;
}

size_t usp_workspace_bytes(const ulysses_shape_t& s, int P_ring) {
    const UspGeom g = usp_geom(s, P_ring);
    // forward: the fp32 running (O, lse) of one query block
    const size_t fwd = g.acc_bytes + g.lse_bytes;
    // backward: fp32 sums of dK and dV over the whole sequence, and the block-pair backward's
    // own workspace (whose fp32 dQ accumulator carries a query block across its pairs)
    const size_t bwd = 2 * align256(size_t(P_ring) * g.kv_elems * 4) + bwd_workspace_bytes(g.sub);
    return fwd > bwd ? fwd : bwd;
}

int launch_usp_fwd(const ulysses_shape_t& s, int P_ring, const MaskArgs& m, float scale, const void* q, const void* k,
                   const void* v, void* o, float* lse, void* ws, cudaStream_t stream) {
    const UspGeom g = usp_geom(s, P_ring);
    char* w = static_cast<char*>(ws);
    float* acc_o = reinterpret_cast<float*>(w);
    float* acc_lse = reinterpret_cast<float*>(w + g.acc_bytes);
    const bool causal = m.kind == ULYSSES_MASK_CAUSAL;
    MaskArgs none{ULYSSES_MASK_NONE, nullptr, nullptr, nullptr, nullptr};
    const __nv_bfloat16* q16 = static_cast<const __nv_bfloat16*>(q);
    const __nv_bfloat16* k16 = static_cast<const __nv_bfloat16*>(k);
    const __nv_bfloat16* v16 = static_cast<const __nv_bfloat16*>(v);
    __nv_bfloat16* o16 = static_cast<__nv_bfloat16*>(o);
    auto pair = [&](int i, int j, cudaStream_t st) {
        const int nj = causal ? i + 1 : P_ring;
        const MaskArgs& mj = (causal && j == i) ? m : none;
        FwdChain ch;
        ch.mode = nj == 1 ? 0 : (j == 0 ? 1 : (j + 1 == nj ? 3 : 2));
        ch.o_acc = acc_o;
        ch.lse_acc = acc_lse;
        return launch_attn_fwd(g.sub, mj, scale, ULYSSES_LAYOUT_TOKEN_SHARDED, q16 + i * g.q_elems, k16 + j * g.kv_elems,
                               v16 + j * g.kv_elems, o16 + i * g.q_elems, lse + i * g.lse_elems, st, ch);
    };
    // Query blocks outer, key blocks inner: a query block's pairs run back to back, merging into
    // the one running pair (stream order keeps each merge after the previous pair's). With a
    // causal mask the first query block has one pair and no running pair. It runs on a side
    // stream beside the others, submitted after the main stream's first launch, so that the block
    // scheduler hands out that launch's CTAs first and the side pair's CTAs fill its last waves.
    SideStream side;
    const bool fork = causal && P_ring > 1 && side_stream(side);
    if (fork && (cudaEventRecord(side.fork, stream) != cudaSuccess ||
                 cudaStreamWaitEvent(side.stream, side.fork, 0) != cudaSuccess))
        return ULYSSES_ERR_CUDA;
    int rc = ULYSSES_OK;
    bool side_done = !fork;
    for (int i = fork ? 1 : 0; rc == ULYSSES_OK && i < P_ring; ++i) {
        const int nj = causal ? i + 1 : P_ring;
        for (int j = 0; rc == ULYSSES_OK && j < nj; ++j) {
            rc = pair(i, j, stream);
            if (rc == ULYSSES_OK && !side_done) {
                side_done = true;
                rc = pair(0, 0, side.stream);
            }
        }
    }
    // the caller's stream waits for the side stream, on error too (a capture must be rejoined)
    if (fork && (cudaEventRecord(side.join, side.stream) != cudaSuccess ||
                 cudaStreamWaitEvent(stream, side.join, 0) != cudaSuccess) && rc == ULYSSES_OK)
        rc = ULYSSES_ERR_CUDA;
    return rc;
}

int launch_usp_bwd(const ulysses_shape_t& s, int P_ring, const MaskArgs& m, float scale, const void* q, const void* k,
                   const void* v, const void* o, const float* lse, const void* dO, void* dq, void* dk, void* dv,
                   void* ws, cudaStream_t stream) {
    const UspGeom g = usp_geom(s, P_ring);
    char* w = static_cast<char*>(ws);
    float* acc_k = reinterpret_cast<float*>(w);
    w += align256(size_t(P_ring) * g.kv_elems * 4);
    float* acc_v = reinterpret_cast<float*>(w);
    w += align256(size_t(P_ring) * g.kv_elems * 4);
    void* sub_ws = w;
    const bool causal = m.kind == ULYSSES_MASK_CAUSAL;
    MaskArgs none{ULYSSES_MASK_NONE, nullptr, nullptr, nullptr, nullptr};
    const __nv_bfloat16* q16 = static_cast<const __nv_bfloat16*>(q);
    const __nv_bfloat16* k16 = static_cast<const __nv_bfloat16*>(k);
    const __nv_bfloat16* v16 = static_cast<const __nv_bfloat16*>(v);
    const __nv_bfloat16* o16 = static_cast<const __nv_bfloat16*>(o);
    const __nv_bfloat16* do16 = static_cast<const __nv_bfloat16*>(dO);
    __nv_bfloat16* dq16 = static_cast<__nv_bfloat16*>(dq);
    __nv_bfloat16* dk16 = static_cast<__nv_bfloat16*>(dk);
    __nv_bfloat16* dv16 = static_cast<__nv_bfloat16*>(dv);
    // block pairs each query block / key block takes part in
    auto q_pairs = [&](int i) { return causal ? i + 1 : P_ring; };
    auto k_pairs = [&](int j) { return causal ? P_ring - j : P_ring; };
    int seen_k[kMaxRing] = {};
    // Query blocks outer, key blocks inner: a query block's pairs run back to back, so its dQ
    // stays in the block-pair backward's fp32 accumulator from the first pair (which zeroes it
    // and computes Delta) to the last (which writes bf16 dQ). dK, dV of a key block are spread
    // over query blocks: its first pair stores them fp32, later pairs add, the last rounds.
    for (int i = 0; i < P_ring; ++i) {
        for (int j = 0; j < q_pairs(i); ++j) {
            const MaskArgs& mj = (causal && j == i) ? m : none;
            BwdChain ch;
            ch.prep = j == 0;
            ch.convert = j + 1 == q_pairs(i);
            const int nk = k_pairs(j), c = seen_k[j]++;
            ch.dkv_mode = nk == 1 ? 0 : (c == 0 ? 1 : (c + 1 == nk ? 3 : 2));
            ch.dk_acc = acc_k + j * g.kv_elems;
            ch.dv_acc = acc_v + j * g.kv_elems;
            int rc = launch_attn_bwd(g.sub, mj, scale, ULYSSES_LAYOUT_TOKEN_SHARDED, q16 + i * g.q_elems,
                                     k16 + j * g.kv_elems, v16 + j * g.kv_elems, o16 + i * g.q_elems,
                                     lse + i * g.lse_elems, do16 + i * g.q_elems, dq16 + i * g.q_elems,
                                     dk16 + j * g.kv_elems, dv16 + j * g.kv_elems, sub_ws, stream, ch);
            if (rc != ULYSSES_OK) return rc;
        }
    }
    return ULYSSES_OK;
}

}  // namespace ulysses
