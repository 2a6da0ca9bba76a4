// Attention forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), one CTA per
// (batch, head, pair of 128-row query tiles).
//
// What it computes (paper summary section 3.4.1 "The challenge at the attention boundary";
// pinyu.ai page "The layout that saves memory breaks at attention"): for one head over the
// full sequence,  S = scale * Q K^T (+ mask),  O = softmax(S) V,  lse = ln sum_j exp(S_ij).
// The softmax is evaluated online over key tiles with a running maximum.
//
// The Ulysses relayouts are fused: the TMA tensor maps address Q, K, V (and the epilogue
// addresses O) in the token-sharded layout [P][B][Lp][H][d], so the "full sequence of
// head h" that a head-group rank would receive from the seq->head all-to-all is only an
// address computation (sender r = s / Lp, local token s % Lp). With the head-sharded
// layout the same kernel reads [P][B][L][Hp][d].
//
// Two query tiles share every K/V tile brought into shared memory, which halves the K/V
// traffic per flop; their softmax warpgroups alternate so that the tensor core works on
// one tile while the other tile's softmax runs. Warp roles (320 threads):
//   warp 0    TMA producer: both Q tiles once, then K and V tiles through their rings;
//   warp 1    MMA issuer: S_t = Q_t K^T into TMEM columns [128 t, 128 t + 128) and
//             O_t += P_t V into [256 + 128 t, ...), with P_t read from the first 64
//             columns of S_t (packed bf16 pairs, the A operand of a TMEM-sourced MMA);
//   warps 2-5 softmax of tile 0, warps 6-9 softmax of tile 1: thread i owns query row i
//             (TMEM lane i): reads S_t in two 64-column halves for the row maximum, then
//             again half by half to write P_t over S_t (keeping the live registers within
//             the 168 a 10-warp CTA allows), rescales O_t in TMEM when the max grows by more
//             than 2^8, and finally normalises and stores O_t and lse.
// The MMA issuer issues PV_t for a key tile before S_t for the next one, and tcgen05
// operations of one thread complete in order: when S_t of a key tile is complete, the
// previous PV_t (which read P_t from the same columns) is too, so O_t may be rescaled and
// the columns reused without a further wait.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "ulysses_internal.h"

namespace ulysses {

struct FwdParams {
    int B, L, H, Hp, Lp, P;
    int G, kv_rep;   // query heads per key/value head; head groups per key/value head copy
    int layout;      // 0 token-sharded, 1 head-sharded
    int n_tiles;     // ceil(L / 128)
    int n_pairs;     // ceil(n_tiles / 2)
    int box_rows;    // rows per TMA box (divides 128; boxes never straddle a shard)
    float scale_log2;
    void* o;
    float* lse;
    const int32_t* rowptr;  // block-sparse CSR over query tiles
    const int32_t* kcols;
    uint32_t* err;
};

// The accumulating kernels' parameters (the Ulysses-ring hybrid's block pairs): a separate
// type, so that the plain kernel's parameters stay as they are.
struct FwdAccParams : FwdParams {
    float* o_acc;    // fp32 running O of the query block (layout of O)
    float* lse_acc;  // running lse (layout of lse)
    int mode;        // 1 store this pair's (O, lse); 2 merge into the running pair; 3 merge, write O and lse
};
template <bool ACC>
using FwdParamsOf = typename std::conditional<ACC, FwdAccParams, FwdParams>::type;

template <int D>
struct FwdCfg {
    static constexpr int NSK = (D == 64) ? 6 : 3;                // K pipeline stages
    static constexpr int NSV = (D == 64) ? 6 : 2;                // V pipeline stages
    static constexpr uint32_t TILE_BYTES = kTile * D * 2;       // one 128-row bf16 tile
    static constexpr uint32_t CHUNK_BYTES = kTile * 128;        // 128 rows x 64 elements
    static constexpr uint32_t OFF_Q = 0;                        // [2] query tiles
    static constexpr uint32_t OFF_K = OFF_Q + 2 * TILE_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + NSK * TILE_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_V + NSV * TILE_BYTES;
    static constexpr uint32_t SMEM_BYTES = OFF_BAR + 512 + 1024;  // + barriers + alignment slack
    static constexpr uint32_t TMEM_COLS = 512;                    // S0 | S1 | O0 | O1
    static constexpr uint32_t kThreads = 320;
};

// Coordinates of global row s of query head h, batch b, in the 5-D map (d, head, row,
// batch, unit): of the query-side tensor, or (KV) of the key/value head that h attends with.
template <bool KV>
__device__ __forceinline__ void qkv_coords(const FwdParams& p, int s, int h, int& c1, int& c2, int& c4) {
    if (p.layout == ULYSSES_LAYOUT_TOKEN_SHARDED) {
        c1 = KV ? h / p.G : h;
        c2 = s % p.Lp;
        c4 = s / p.Lp;  // == P past the end of the sequence: out of bounds, filled with zeros
    } else {
        // head group g holds key/value heads [g Hkvp, (g + 1) Hkvp), or one copy of head g / kv_rep
        c1 = KV ? (p.kv_rep == 1 ? (h % p.Hp) / p.G : 0) : h % p.Hp;
        c2 = s;
        c4 = h / p.Hp;
    }
}

// Loads rows [s0, s0 + 128) of query head h (KV: of its key/value head) into a tile of D/64
// swizzled chunks of 128 x 64.
template <int D, bool KV>
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, const FwdParams& p,
                                          int s0, int h, int b) {
    for (int c = 0; c < D / 64; ++c) {
        for (int r = 0; r < kTile; r += p.box_rows) {
            int c1, c2, c4;
            qkv_coords<KV>(p, s0 + r, h, c1, c2, c4);
            tma_load_5d(dst + c * FwdCfg<D>::CHUNK_BYTES + r * 128, map, bar, c * 64, c1, c2, b, c4);
        }
    }
}

// Key tiles of one query tile, in ascending order.
template <int MASK>
struct TileList {
    int n, first;
    const int32_t* cols;
    __device__ __forceinline__ void init(const FwdParams& p, int qt, bool exists) {
        cols = p.kcols;
        first = 0;
        if (!exists) n = 0;
        else if (MASK == ULYSSES_MASK_CAUSAL) n = qt + 1;
        else if (MASK == ULYSSES_MASK_NONE) n = p.n_tiles;
        else { first = p.rowptr[qt]; n = p.rowptr[qt + 1] - first; }
    }
    __device__ __forceinline__ int kt(int c) const {
        return MASK == ULYSSES_MASK_BLOCK_SPARSE ? cols[first + c] : c;
    }
};

// The merged, ascending key-tile sequence of the CTA's two query tiles: each step names a
// key tile and which of the two tiles use it.
template <int MASK>
struct PairSeq {
    TileList<MASK> t0, t1;
    int c0, c1;
    __device__ __forceinline__ void init(const FwdParams& p, int qt0, bool has1) {
        t0.init(p, qt0, true);
        t1.init(p, qt0 + 1, has1);
        c0 = c1 = 0;
    }
    // returns false when both lists are exhausted
    __device__ __forceinline__ bool next(int& kt, bool& in0, bool& in1) {
        const bool a0 = c0 < t0.n, a1 = c1 < t1.n;
        if (!a0 && !a1) return false;
        const int k0 = a0 ? t0.kt(c0) : 0x7fffffff;
        const int k1 = a1 ? t1.kt(c1) : 0x7fffffff;
        kt = k0 < k1 ? k0 : k1;
        in0 = a0 && k0 == kt;
        in1 = a1 && k1 == kt;
        c0 += in0;
        c1 += in1;
        return true;
    }
};

// ACC: the epilogue merges this launch's normalised (O, lse) into an fp32 running pair
// (the online-softmax merge of the Ulysses-ring hybrid's block pairs) instead of storing it
template <int D, int MASK, bool ACC>
__global__ void __launch_bounds__(320, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const FwdParamsOf<ACC> p) {
    using C = FwdCfg<D>;
    constexpr int NSK = C::NSK;
    constexpr int NSV = C::NSV;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + C::OFF_Q;
    uint8_t* sK = smem + C::OFF_K;
    uint8_t* sV = smem + C::OFF_V;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* q_full = bars + 0;
    uint64_t* k_full = bars + 1;            // [NSK]
    uint64_t* k_empty = k_full + NSK;       // [NSK]
    uint64_t* v_full = k_empty + NSK;       // [NSV]
    uint64_t* v_empty = v_full + NSV;       // [NSV]
    uint64_t* s_full = v_empty + NSV;       // [2]
    uint64_t* p_full = s_full + 2;          // [2]
    uint64_t* o_done = p_full + 2;
    uint64_t* drain = o_done + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = static_cast<int>(warp_id());
    const int lane = static_cast<int>(lane_id());
    // Query-tile pairs vary fastest. With a causal mask grid row y holds a group of G heads
    // (G = gridDim.x / n_pairs, chosen so that their K and V fit in a quarter of L2), dealt
    // out heaviest pair first across the group: the resident CTAs share a few heads' K, V in
    // L2, and the light pairs of every group fill the last waves instead of a lone head's.
    int bh = blockIdx.y, pair = blockIdx.x;
    if (MASK == ULYSSES_MASK_CAUSAL) {
        const int G = static_cast<int>(gridDim.x) / p.n_pairs;
        const int Gg = min(G, p.B * p.H - static_cast<int>(blockIdx.y) * G);
        const int r = static_cast<int>(blockIdx.x);
        if (r >= Gg * p.n_pairs) return;  // the last group's spare CTAs (all threads leave)
        pair = p.n_pairs - 1 - r / Gg;
        bh = static_cast<int>(blockIdx.y) * G + r % Gg;
    }
    const int b = bh / p.H;
    const int h = bh % p.H;
    const int qt0 = 2 * pair;
    const bool has1 = qt0 + 1 < p.n_tiles;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < NSK; ++i) {
            mbar_init(k_full + i, 1);
            mbar_init(k_empty + i, 1);
        }
        for (int i = 0; i < NSV; ++i) {
            mbar_init(v_full + i, 1);
            mbar_init(v_empty + i, 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(s_full + t, 1);
            mbar_init(p_full + t, 4);
        }
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Abort ab{abort_flag, p.err, KID_FWD};
    if (warp < 2) {
      if (warp == 0) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            PairSeq<MASK> seq;
            seq.init(p, qt0, has1);
            int nk = 0, nv = 0;  // loads issued so far, per tensor
            bool ok = true;
            bool any = false;
            int kt;
            bool in0, in1;
            for (int j = 0; seq.next(kt, in0, in1); ++j) {
                if (!any) {
                    any = true;
                    mbar_arrive_expect_tx(q_full, 2 * C::TILE_BYTES);
                    load_tile<D, false>(sQ, &tm_q, q_full, p, qt0 * kTile, h, b);
                    load_tile<D, false>(sQ + C::TILE_BYTES, &tm_q, q_full, p, (qt0 + 1) * kTile, h, b);
                }
                const int sk = j % NSK, sv = j % NSV;
                if (j >= NSK && !(ok = mbar_wait(k_empty + sk, ((j / NSK) - 1) & 1, ab, ROLE_LOAD, 1))) break;
                mbar_arrive_expect_tx(k_full + sk, C::TILE_BYTES);
                load_tile<D, true>(sK + sk * C::TILE_BYTES, &tm_k, k_full + sk, p, kt * kTile, h, b);
                ++nk;
                if (j >= NSV && !(ok = mbar_wait(v_empty + sv, ((j / NSV) - 1) & 1, ab, ROLE_LOAD, 2))) break;
                mbar_arrive_expect_tx(v_full + sv, C::TILE_BYTES);
                load_tile<D, true>(sV + sv * C::TILE_BYTES, &tm_v, v_full + sv, p, kt * kTile, h, b);
                ++nv;
            }
            if (!ok) {
                // let copies already in flight land before the CTA can exit
                mbar_drain(q_full, 0);
                for (int st = 0; st < NSK; ++st) {
                    const int ck = nk > st ? (nk - 1 - st) / NSK + 1 : 0;  // K loads issued to stage st
                    if (ck > 0) mbar_drain(k_full + st, (ck - 1) & 1);
                }
                for (int st = 0; st < NSV; ++st) {
                    const int cv = nv > st ? (nv - 1 - st) / NSV + 1 : 0;
                    if (cv > 0) mbar_drain(v_full + st, (cv - 1) & 1);
                }
            }
        }
      } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t idO = idesc_bf16(128, D, 0, 1);
            const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
            PairSeq<MASK> seq;
            seq.init(p, qt0, has1);
            int kt, nkt;
            bool in0, in1, nin0 = false, nin1 = false;
            bool ok = true;
            bool cur = seq.next(kt, in0, in1);
            // S_t = Q_t K^T for the key tile in K stage sk
            auto issue_s = [&](int t, int sk) {
                const uint64_t dq = sdesc_sw128(aQ + t * C::TILE_BYTES, 16, 1024);
                const uint64_t dk = sdesc_sw128(aK + sk * C::TILE_BYTES, 16, 1024);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k >> 2) * C::CHUNK_BYTES + (k & 3) * 32;
                    umma_ss(tmem + 128 * t, sdesc_add(dq, off), sdesc_add(dk, off), idS, k > 0 ? 1u : 0u);
                }
                umma_commit(s_full + t);
            };
            // O_t += P_t V for the value tile in V stage sv
            auto issue_pv = [&](int t, int sv, bool first) {
                const uint64_t dv = sdesc_sw128(aV + sv * C::TILE_BYTES, C::CHUNK_BYTES, 1024);
#pragma unroll
                for (int k = 0; k < kTile / 16; ++k)  // 16 keys = 8 TMEM columns of P per step
                    umma_ts(tmem + 256 + 128 * t, tmem + 128 * t + k * 8, sdesc_add(dv, k * 2048), idO,
                            (!first || k > 0) ? 1u : 0u);
            };
            if (cur) {
                ok = mbar_wait(q_full, 0, ab, ROLE_MMA, 1) && mbar_wait(k_full, 0, ab, ROLE_MMA, 2);
                if (ok) {
                    tc_fence_after();
                    if (in0) issue_s(0, 0);
                    if (in1) issue_s(1, 0);
                    umma_commit(k_empty);
                }
            }
            int c0 = 0, c1 = 0;  // PV MMAs issued per tile
            for (int j = 0; ok && cur; ++j) {
                const bool nxt = seq.next(nkt, nin0, nin1);
                const int sv = j % NSV, skn = (j + 1) % NSK;
                if (!(ok = mbar_wait(v_full + sv, (j / NSV) & 1, ab, ROLE_MMA, 3))) break;
                if (in0) {
                    if (!(ok = mbar_wait(p_full, c0 & 1, ab, ROLE_MMA, 4))) break;
                    tc_fence_after();
                    issue_pv(0, sv, c0 == 0);
                    ++c0;
                }
                if (nxt) {
                    if (!(ok = mbar_wait(k_full + skn, ((j + 1) / NSK) & 1, ab, ROLE_MMA, 5))) break;
                    tc_fence_after();
                    if (nin0) issue_s(0, skn);
                }
                if (in1) {
                    if (!(ok = mbar_wait(p_full + 1, c1 & 1, ab, ROLE_MMA, 6))) break;
                    tc_fence_after();
                    issue_pv(1, sv, c1 == 0);
                    ++c1;
                }
                if (nxt) {
                    if (nin1) issue_s(1, skn);
                    umma_commit(k_empty + skn);
                }
                umma_commit(v_empty + sv);
                cur = nxt;
                kt = nkt;
                in0 = nin0;
                in1 = nin1;
            }
            if (ok) umma_commit(o_done);
            else {
                umma_commit(drain);
                mbar_drain(drain, 0);
            }
        }
      }
    } else {
        // ------------------------------------------------------------------ softmax (tile t)
        const int t = warp < 6 ? 0 : 1;
        const int wq = warp & 3;                  // TMEM lane quadrant of this warp
        const int row = wq * 32 + lane;           // query row within the tile (TMEM lane)
        const uint32_t lane_off = uint32_t(wq * 32) << 16;
        const int qt = qt0 + t;
        const int s_row = qt * kTile + row;       // global query index
        const uint32_t tS = tmem + 128 * t;
        const uint32_t tO = tmem + 256 + 128 * t;
        TileList<MASK> list;
        list.init(p, qt, t == 0 || has1);
        float m_used = -INFINITY;                 // running max, log2 domain
        float l_sum = 0.f;
        bool ok = true;
        for (int c = 0; c < list.n; ++c) {
            const int kt = list.kt(c);
            ok = __all_sync(0xffffffffu, mbar_wait(s_full + t, c & 1, ab, ROLE_SOFTMAX, 1));
            if (!ok) break;
            tc_fence_after();
            const int k0 = kt * kTile;
            const bool diag = (MASK == ULYSSES_MASK_CAUSAL) && (kt == qt);
            const bool masked = diag || (k0 + kTile > p.L);
            // keys past the diagonal (causal) or past the end of the sequence are excluded
            auto mask_half = [&](float* v, int c0) {
                if (masked) {
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        const int key = k0 + c0 + i;
                        if ((diag && key > s_row) || key >= p.L) v[i] = -INFINITY;
                    }
                }
            };
            // pass 1: row maximum
            float mx = -INFINITY;
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                float v[64];
                tmem_ld32(tS + lane_off + hh * 64, v);
                tmem_ld32(tS + lane_off + hh * 64 + 32, v + 32);
                tmem_wait_ld();
                mask_half(v, hh * 64);
#pragma unroll
                for (int i = 0; i < 64; ++i) mx = fmaxf(mx, v[i]);
            }
            const float m_new = fmaxf(m_used, mx * p.scale_log2);
            const bool need = m_new > m_used + 8.0f;
            const float alpha = need ? ex2(m_used - m_new) : 1.0f;  // ex2(-inf) = 0 for a first max
            if (need) m_used = m_new;
            const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
            // pass 2: P = 2^(S*scale*log2e - m) as bf16 pairs over the first 64 columns of S_t
            // (half hh of S lands in columns [32 hh, 32 hh + 32), already read)
            float rs = 0.f;
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                float v[64];
                tmem_ld32(tS + lane_off + hh * 64, v);
                tmem_ld32(tS + lane_off + hh * 64 + 32, v + 32);
                tmem_wait_ld();
                mask_half(v, hh * 64);
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float e0 = ex2(fmaf(v[2 * i], p.scale_log2, neg_m));
                    const float e1 = ex2(fmaf(v[2 * i + 1], p.scale_log2, neg_m));
                    rs += e0 + e1;
                    pk[i] = pack_bf16(e0, e1);
                }
                tmem_st32_u(tS + lane_off + hh * 32, pk);
            }
            l_sum = l_sum * alpha + rs;
            // O_t is stable (the previous PV_t was issued before this S_t and has completed);
            // rescale it before this step's PV_t, which waits for the arrival below
            if (c > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll 1
                for (int i = 0; i < D / 32; ++i) {
                    float o[32];
                    tmem_ld32(tO + lane_off + i * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int x = 0; x < 32; ++x) o[x] *= alpha;
                    tmem_st32(tO + lane_off + i * 32, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full + t);
        }

        // ------------------------------------------------------------------ epilogue
        if (ok && list.n > 0) ok = __all_sync(0xffffffffu, mbar_wait(o_done, 0, ab, ROLE_EPI, 1));
        if (ok) {
            tc_fence_after();
            const bool valid = s_row < p.L;
            const bool any_key = l_sum > 0.f;
            const float inv_l = any_key ? 1.0f / l_sum : 0.f;
            size_t orow_off;
            if (p.layout == ULYSSES_LAYOUT_TOKEN_SHARDED) {
                const int r = s_row / p.Lp, tt = s_row % p.Lp;
                orow_off = ((size_t(r) * p.B + b) * p.Lp + tt) * size_t(p.H) * D + size_t(h) * D;
            } else {
                const int g = h / p.Hp, j = h % p.Hp;
                orow_off = ((size_t(g) * p.B + b) * p.L + s_row) * size_t(p.Hp) * D + size_t(j) * D;
            }
            __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.o) + orow_off;
            const size_t li = ((size_t(h / p.Hp) * p.B + b) * p.Hp + (h % p.Hp)) * p.L + s_row;
            float lse = any_key ? (m_used + log2f(l_sum)) * 0.69314718055994531f : -INFINITY;
            // ACC: this pair's part gets weight w_new, the running part w_run (lse = ln sum exp)
            float w_run = 0.f, w_new = 1.f;
            int mode = 0;
            float* arow = nullptr;
            if constexpr (ACC) {
                mode = p.mode;
                arow = p.o_acc + orow_off;
                if (mode >= 2 && valid) {
                    const float lr = p.lse_acc[li];
                    const float mx = fmaxf(lr, lse);
                    if (mx == -INFINITY) {
                        w_new = 0.f;
                    } else {
                        const float er = __expf(lr - mx), en = __expf(lse - mx);
                        const float tot = er + en;
                        w_run = er / tot;
                        w_new = en / tot;
                        lse = mx + __logf(tot);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < D / 32; ++i) {
                float o[32];
                if (list.n > 0) {
                    tmem_ld32(tO + lane_off + i * 32, o);
                    tmem_wait_ld();
                }
#pragma unroll
                for (int x = 0; x < 32; ++x) o[x] = (list.n > 0) ? o[x] * inv_l : 0.f;
                if (!valid) continue;
                if (ACC && mode != 0) {
                    float4* a4 = reinterpret_cast<float4*>(arow + i * 32);
                    if (mode >= 2) {
#pragma unroll
                        for (int y = 0; y < 8; ++y) {
                            const float4 t = a4[y];
                            o[4 * y] = w_run * t.x + w_new * o[4 * y];
                            o[4 * y + 1] = w_run * t.y + w_new * o[4 * y + 1];
                            o[4 * y + 2] = w_run * t.z + w_new * o[4 * y + 2];
                            o[4 * y + 3] = w_run * t.w + w_new * o[4 * y + 3];
                        }
                    }
                    if (mode <= 2) {
#pragma unroll
                        for (int y = 0; y < 8; ++y) a4[y] = make_float4(o[4 * y], o[4 * y + 1], o[4 * y + 2], o[4 * y + 3]);
                        continue;
                    }
                }
                uint4* dst = reinterpret_cast<uint4*>(orow + i * 32);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    dst[v] = make_uint4(pack_bf16(o[8 * v + 0], o[8 * v + 1]), pack_bf16(o[8 * v + 2], o[8 * v + 3]),
                                        pack_bf16(o[8 * v + 4], o[8 * v + 5]), pack_bf16(o[8 * v + 6], o[8 * v + 7]));
                }
            }
            if (valid) {
                if (ACC && mode != 0 && mode <= 2) {
                    if constexpr (ACC) p.lse_acc[li] = lse;
                } else {
                    p.lse[li] = lse;
                }
            }
        }
    }

    tc_fence_before();
    __syncwarp();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int D, int MASK, bool ACC>
static int launch_fwd_t(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                        const FwdParamsOf<ACC>& p, cudaStream_t stream) {
    using C = FwdCfg<D>;
    auto kern = attn_fwd_kernel<D, MASK, ACC>;
    if (!set_max_dynamic_smem(reinterpret_cast<const void*>(kern), C::SMEM_BYTES)) return ULYSSES_ERR_CUDA;
    const int bh = p.B * p.H;
    int G = 1;
    if (MASK == ULYSSES_MASK_CAUSAL) {
        const size_t kv_head = size_t(4) * size_t(p.L) * D;  // K and V of one head, bf16
        G = int(std::min<size_t>(size_t(bh), std::max<size_t>(1, (size_t(32) << 20) / kv_head)));
    }
    dim3 grid(G * p.n_pairs, (bh + G - 1) / G);
    kern<<<grid, C::kThreads, C::SMEM_BYTES, stream>>>(mq, mk, mv, p);
    return cudaGetLastError() == cudaSuccess ? ULYSSES_OK : ULYSSES_ERR_CUDA;
}

template <int D>
static int launch_fwd_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const FwdParams& p,
                        int kind, const FwdChain& chain, cudaStream_t stream) {
    if (chain.mode != 0) {
        FwdAccParams ap;
        static_cast<FwdParams&>(ap) = p;
        ap.o_acc = chain.o_acc;
        ap.lse_acc = chain.lse_acc;
        ap.mode = chain.mode;
        // the accumulating epilogue is built for the masks of the ring blocks only
        if (kind == ULYSSES_MASK_CAUSAL) return launch_fwd_t<D, ULYSSES_MASK_CAUSAL, true>(mq, mk, mv, ap, stream);
        if (kind == ULYSSES_MASK_NONE) return launch_fwd_t<D, ULYSSES_MASK_NONE, true>(mq, mk, mv, ap, stream);
        return ULYSSES_ERR_UNSUPPORTED;
    }
    if (kind == ULYSSES_MASK_CAUSAL) return launch_fwd_t<D, ULYSSES_MASK_CAUSAL, false>(mq, mk, mv, p, stream);
    if (kind == ULYSSES_MASK_NONE) return launch_fwd_t<D, ULYSSES_MASK_NONE, false>(mq, mk, mv, p, stream);
    return launch_fwd_t<D, ULYSSES_MASK_BLOCK_SPARSE, false>(mq, mk, mv, p, stream);
}

int launch_attn_fwd(const ulysses_shape_t& s, const MaskArgs& m, float scale, int layout, const void* q,
                    const void* k, const void* v, void* o, float* lse, cudaStream_t stream, const FwdChain& chain) {
    FwdParams p{};
    p.B = s.B; p.L = s.L; p.H = s.H; p.P = s.P; p.Hp = s.H / s.P; p.Lp = s.L / s.P;
    const KvInfo kv = kv_info(s);
    p.G = kv.G;
    p.kv_rep = kv.rep;
    p.layout = layout;
    p.n_tiles = (s.L + kTile - 1) / kTile;
    p.n_pairs = (p.n_tiles + 1) / 2;
    p.box_rows = layout == ULYSSES_LAYOUT_TOKEN_SHARDED ? gcd_int(p.Lp, kTile) : kTile;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.o = o;
    p.lse = lse;
    p.rowptr = m.q_rowptr;
    p.kcols = m.q_kcols;
    p.err = device_error_word();
    if (!p.err) return ULYSSES_ERR_CUDA;
    CUtensorMap mq, mk, mv;
    if (!encode_qkv_map(&mq, q, s, layout, p.box_rows, s.H, s.H / s.P) ||
        !encode_qkv_map(&mk, k, s, layout, p.box_rows, kv.Hkv, kv.Hkvp) ||
        !encode_qkv_map(&mv, v, s, layout, p.box_rows, kv.Hkv, kv.Hkvp))
        return ULYSSES_ERR_CUDA;
    if (chain.mode < 0 || chain.mode > 3 || (chain.mode != 0 && (!chain.o_acc || !chain.lse_acc)))
        return ULYSSES_ERR_INVALID_ARG;
    if (s.d_h == 128) return launch_fwd_d<128>(mq, mk, mv, p, m.kind, chain, stream);
    return launch_fwd_d<64>(mq, mk, mv, p, m.kind, chain, stream);
}

}  // namespace ulysses
