// Ulysses-ring hybrid ("USP" on the aifetchly page, step 5; Ring Attention in the reading
// notes, section 5.2): P = P_u x P_ring shards. The sequence is cut into P_ring contiguous ring
// blocks of L / P_ring tokens; each block is itself a token-sharded tensor of P_u = P / P_ring
// shards, inside which the Ulysses relayout spreads the H heads over P_u head groups (so only
// P_u, not P, must divide H). Across blocks, the key/value blocks are streamed past each query
// block and the per-block attention results are merged with the online-softmax rule:
//   m = max_j lse_j,  lse = m + ln sum_j exp(lse_j - m),  O = sum_j exp(lse_j - lse) O_j.
// The block-pair attentions are the library's own forward and backward on tensor slices: causal
// on the diagonal block pair and dense on every pair below it (on all pairs for a dense mask). The
// backward of a block pair uses the merged O and lse, so its probabilities are those of the
// whole row; its partial gradients are summed over block pairs in fp32 inside the block-pair
// backward (its dQ accumulator, and an fp32 store/add mode of its dK, dV epilogue).
#include "common.cuh"
#include "ulysses_internal.h"

namespace ulysses {

// Merge of n partial results per (row, head): o_parts[j] [Pu][B][Lp][H][d] bf16 and lse_parts[j]
// [Pu][B][H/Pu][Lb] fp32 (the layouts of one ring block) into o, lse of the same layouts.
// Eight lanes per (row, head), each with d/8 elements.
struct MergeArgs {
    const __nv_bfloat16* o_parts[kMaxRing];
    const float* lse_parts[kMaxRing];
    int n;
    __nv_bfloat16* o;
    float* lse;
    int Pu, B, Lp, H, Hp, Lb, d;
};

template <int D>
__global__ void __launch_bounds__(256) usp_merge_kernel(MergeArgs a) {
    constexpr int LPR = 8, EPT = D / LPR;  // lanes per (row, head), elements per lane
    const size_t items = size_t(a.Pu) * a.B * a.Lp * a.H;
    const int sub = threadIdx.x % LPR;
    for (size_t it = (size_t(blockIdx.x) * blockDim.x + threadIdx.x) / LPR; it < items;
         it += size_t(gridDim.x) * blockDim.x / LPR) {
        // item = ((r * B + b) * Lp + t) * H + h, the token-sharded row order
        const int h = int(it % a.H);
        const size_t row = it / a.H;
        const int t = int(row % a.Lp);
        const int b = int((row / a.Lp) % a.B);
        const int r = int(row / (size_t(a.Lp) * a.B));
        const int s = r * a.Lp + t;                  // token within the block
        const int g = h / a.Hp, j = h % a.Hp;
        const size_t li = ((size_t(g) * a.B + b) * a.Hp + j) * a.Lb + s;
        float m = -INFINITY;
        for (int p = 0; p < a.n; ++p) m = fmaxf(m, a.lse_parts[p][li]);
        float acc[EPT];
#pragma unroll
        for (int e = 0; e < EPT; ++e) acc[e] = 0.f;
        float tot = 0.f;
        if (m != -INFINITY) {
            for (int p = 0; p < a.n; ++p) {
                const float w = __expf(a.lse_parts[p][li] - m);
                tot += w;
                const uint4* src = reinterpret_cast<const uint4*>(a.o_parts[p] + it * D + sub * EPT);
#pragma unroll
                for (int v = 0; v < EPT / 8; ++v) {
                    const uint4 x = src[v];
                    const __nv_bfloat162* x2 = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = __bfloat1622float2(x2[i]);
                        acc[8 * v + 2 * i] = fmaf(w, f.x, acc[8 * v + 2 * i]);
                        acc[8 * v + 2 * i + 1] = fmaf(w, f.y, acc[8 * v + 2 * i + 1]);
                    }
                }
            }
        }
        const float inv = tot > 0.f ? 1.f / tot : 0.f;
        uint4* dst = reinterpret_cast<uint4*>(a.o + it * D + sub * EPT);
#pragma unroll
        for (int v = 0; v < EPT / 8; ++v)
            dst[v] = make_uint4(pack_bf16(acc[8 * v] * inv, acc[8 * v + 1] * inv),
                                pack_bf16(acc[8 * v + 2] * inv, acc[8 * v + 3] * inv),
                                pack_bf16(acc[8 * v + 4] * inv, acc[8 * v + 5] * inv),
                                pack_bf16(acc[8 * v + 6] * inv, acc[8 * v + 7] * inv));
        if (sub == 0) a.lse[li] = m == -INFINITY ? -INFINITY : m + __logf(tot);
    }
}

namespace {

unsigned grid_for(size_t work, int per_block) {
    size_t blocks = (work + per_block - 1) / per_block;
    const size_t cap = size_t(device_sm_count()) * 16;
    if (blocks > cap) blocks = cap;
    return unsigned(blocks ? blocks : 1);
}

struct UspGeom {
    ulysses_shape_t sub;    // one ring block: L / P_ring tokens, P / P_ring shards
    size_t q_elems, kv_elems, lse_elems;  // per ring block
    size_t part_bytes, lse_bytes;         // one partial O (bf16) and lse (fp32), 256-aligned
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
    g.part_bytes = align256(g.q_elems * 2);
    g.lse_bytes = align256(g.lse_elems * 4);
    return g;
}

}  // namespace

size_t usp_workspace_bytes(const ulysses_shape_t& s, int P_ring) {
    const UspGeom g = usp_geom(s, P_ring);
    // forward: up to P_ring partial (O, lse) of one query block
    const size_t fwd = size_t(P_ring) * (g.part_bytes + g.lse_bytes);
    // backward: fp32 sums of dK and dV over the whole sequence, and the block-pair backward's
    // own workspace (whose fp32 dQ accumulator carries a query block across its pairs)
    const size_t bwd = 2 * align256(size_t(P_ring) * g.kv_elems * 4) + bwd_workspace_bytes(g.sub);
    return fwd > bwd ? fwd : bwd;
}

int launch_usp_fwd(const ulysses_shape_t& s, int P_ring, const MaskArgs& m, float scale, const void* q, const void* k,
                   const void* v, void* o, float* lse, void* ws, cudaStream_t stream) {
    const UspGeom g = usp_geom(s, P_ring);
    char* w = static_cast<char*>(ws);
    char* parts_o = w;
    char* parts_lse = parts_o + size_t(P_ring) * g.part_bytes;
    const bool causal = m.kind == ULYSSES_MASK_CAUSAL;
    MaskArgs none{ULYSSES_MASK_NONE, nullptr, nullptr, nullptr, nullptr};
    const __nv_bfloat16* q16 = static_cast<const __nv_bfloat16*>(q);
    const __nv_bfloat16* k16 = static_cast<const __nv_bfloat16*>(k);
    const __nv_bfloat16* v16 = static_cast<const __nv_bfloat16*>(v);
    for (int i = 0; i < P_ring; ++i) {
        const int nj = causal ? i + 1 : P_ring;
        MergeArgs a{};
        for (int j = 0; j < nj; ++j) {
            void* po = parts_o + size_t(j) * g.part_bytes;
            float* pl = reinterpret_cast<float*>(parts_lse + size_t(j) * g.lse_bytes);
            const MaskArgs& mj = (causal && j == i) ? m : none;
            int rc = launch_attn_fwd(g.sub, mj, scale, ULYSSES_LAYOUT_TOKEN_SHARDED, q16 + i * g.q_elems,
                                     k16 + j * g.kv_elems, v16 + j * g.kv_elems, po, pl, stream);
            if (rc != ULYSSES_OK) return rc;
            a.o_parts[j] = static_cast<const __nv_bfloat16*>(po);
            a.lse_parts[j] = pl;
        }
        a.n = nj;
        a.o = static_cast<__nv_bfloat16*>(o) + i * g.q_elems;
        a.lse = lse + i * g.lse_elems;
        a.Pu = g.sub.P; a.B = s.B; a.Lp = g.sub.L / g.sub.P; a.H = s.H; a.Hp = s.H / g.sub.P; a.Lb = g.sub.L;
        a.d = s.d_h;
        const size_t items = size_t(s.B) * g.sub.L * s.H;
        if (s.d_h == 128) usp_merge_kernel<128><<<grid_for(items * 8, 256), 256, 0, stream>>>(a);
        else usp_merge_kernel<64><<<grid_for(items * 8, 256), 256, 0, stream>>>(a);
        if (cudaGetLastError() != cudaSuccess) return ULYSSES_ERR_CUDA;
        // the next query block reuses the partial buffers after this merge (stream order)
    }
    return ULYSSES_OK;
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
