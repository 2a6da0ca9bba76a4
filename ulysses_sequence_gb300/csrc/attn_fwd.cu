// Attention forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), one CTA per
// (batch, head, 128-row query tile).
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
// Warp roles (192 threads):
//   warp 0   TMA producer: Q once, then K and V tiles through an NS-stage ring;
//   warp 1   MMA issuer: S = Q K^T into TMEM columns [0,128); O += P V into [128,128+d)
//            with P read from TMEM columns [256,320) (the A operand of a TMEM-sourced MMA);
//   warps 2-5 softmax: thread i owns query row i (TMEM lane i): reads S from TMEM, masks,
//            updates the running max and sum, writes P as packed bf16 pairs into TMEM,
//            rescales O in TMEM when the max grows by more than 2^8, and finally
//            normalises and stores O and lse.
// Keeping P in tensor memory leaves shared memory to the Q tile and three K/V stages, and
// takes the P traffic off the shared-memory port that the MMA operand reads saturate.
#include "common.cuh"
#include "ulysses_internal.h"

namespace ulysses {

struct FwdParams {
    int B, L, H, Hp, Lp, P;
    int layout;      // 0 token-sharded, 1 head-sharded
    int n_tiles;     // ceil(L / 128)
    int box_rows;    // rows per TMA box (divides 128; boxes never straddle a shard)
    float scale_log2;
    void* o;
    float* lse;
    const int32_t* rowptr;  // block-sparse CSR over query tiles
    const int32_t* kcols;
    uint32_t* err;
};

template <int D>
struct FwdCfg {
    static constexpr int NS = (D == 64) ? 6 : 3;                 // K/V pipeline stages
    static constexpr uint32_t TILE_BYTES = kTile * D * 2;       // one 128-row bf16 tile
    static constexpr uint32_t CHUNK_BYTES = kTile * 128;        // 128 rows x 64 elements
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + TILE_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + NS * TILE_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_V + NS * TILE_BYTES;
    static constexpr uint32_t SMEM_BYTES = OFF_BAR + 256 + 1024;  // + barriers + alignment slack
    static constexpr uint32_t TMEM_COLS = 512;                    // S 128 | O 128 | P 64 (bf16 pairs)
    static constexpr uint32_t T_S = 0, T_O = 128, T_P = 256;
};

// Coordinates of global row s of head h, batch b, in the 5-D map (d, head, row, batch, unit).
__device__ __forceinline__ void qkv_coords(const FwdParams& p, int s, int h, int& c1, int& c2, int& c4) {
    if (p.layout == ULYSSES_LAYOUT_TOKEN_SHARDED) {
        c1 = h;
        c2 = s % p.Lp;
        c4 = s / p.Lp;  // == P past the end of the sequence: out of bounds, filled with zeros
    } else {
        c1 = h % p.Hp;
        c2 = s;
        c4 = h / p.Hp;
    }
}

// Loads rows [s0, s0 + 128) of head h into a tile of D/64 swizzled chunks of 128 x 64.
template <int D>
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, const FwdParams& p,
                                          int s0, int h, int b) {
    for (int c = 0; c < D / 64; ++c) {
        for (int r = 0; r < kTile; r += p.box_rows) {
            int c1, c2, c4;
            qkv_coords(p, s0 + r, h, c1, c2, c4);
            tma_load_5d(dst + c * FwdCfg<D>::CHUNK_BYTES + r * 128, map, bar, c * 64, c1, c2, b, c4);
        }
    }
}

template <int MASK>
__device__ __forceinline__ int fwd_kv_count(const FwdParams& p, int qt, int& first) {
    if (MASK == ULYSSES_MASK_CAUSAL) { first = 0; return qt + 1; }
    if (MASK == ULYSSES_MASK_NONE) { first = 0; return p.n_tiles; }
    first = p.rowptr[qt];
    return p.rowptr[qt + 1] - first;
}

template <int MASK>
__device__ __forceinline__ int fwd_kv_tile(const FwdParams& p, int first, int it) {
    if (MASK == ULYSSES_MASK_BLOCK_SPARSE) return p.kcols[first + it];
    return it;
}

template <int D, int MASK>
__global__ void __launch_bounds__(192, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    using C = FwdCfg<D>;
    constexpr int NS = C::NS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + C::OFF_Q;
    uint8_t* sK = smem + C::OFF_K;
    uint8_t* sV = smem + C::OFF_V;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* q_full = bars + 0;
    uint64_t* k_full = bars + 1;            // [NS]
    uint64_t* k_empty = k_full + NS;        // [NS]
    uint64_t* v_full = k_empty + NS;        // [NS]
    uint64_t* v_empty = v_full + NS;        // [NS]
    uint64_t* s_full = v_empty + NS;
    uint64_t* s_free = s_full + 1;
    uint64_t* p_full = s_free + 1;
    uint64_t* pv_done = p_full + 1;
    uint64_t* drain = pv_done + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = static_cast<int>(warp_id());
    const int lane = static_cast<int>(lane_id());
    // query tiles vary fastest (heaviest causal tiles first), so the CTAs resident at one
    // time share one head and its K, V stay in L2
    const int bh = blockIdx.y;
    const int b = bh / p.H;
    const int h = bh % p.H;
    const int qt = (MASK == ULYSSES_MASK_CAUSAL) ? (p.n_tiles - 1 - static_cast<int>(blockIdx.x))
                                                  : static_cast<int>(blockIdx.x);
    int kv_first = 0;
    const int n_kv = fwd_kv_count<MASK>(p, qt, kv_first);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < NS; ++i) {
            mbar_init(k_full + i, 1);
            mbar_init(k_empty + i, 1);
            mbar_init(v_full + i, 1);
            mbar_init(v_empty + i, 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_free, 4);
        mbar_init(p_full, 4);
        mbar_init(pv_done, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem + C::T_S;
    const uint32_t tO = tmem + C::T_O;
    const uint32_t tP = tmem + C::T_P;
    const Abort ab{abort_flag, p.err, KID_FWD};

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        if (lane == 0 && n_kv > 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            int nk = 0, nv = 0;  // loads issued so far, per tensor
            bool ok = true;
            mbar_arrive_expect_tx(q_full, C::TILE_BYTES);
            load_tile<D>(sQ, &tm_q, q_full, p, qt * kTile, h, b);
            for (int it = 0; it < n_kv; ++it) {
                const int st = it % NS;
                const uint32_t ph = (it / NS) & 1;
                const int kt = fwd_kv_tile<MASK>(p, kv_first, it);
                if (it >= NS && !(ok = mbar_wait(k_empty + st, ph ^ 1, ab, ROLE_LOAD, 1))) break;
                mbar_arrive_expect_tx(k_full + st, C::TILE_BYTES);
                load_tile<D>(sK + st * C::TILE_BYTES, &tm_k, k_full + st, p, kt * kTile, h, b);
                ++nk;
                if (it >= NS && !(ok = mbar_wait(v_empty + st, ph ^ 1, ab, ROLE_LOAD, 2))) break;
                mbar_arrive_expect_tx(v_full + st, C::TILE_BYTES);
                load_tile<D>(sV + st * C::TILE_BYTES, &tm_v, v_full + st, p, kt * kTile, h, b);
                ++nv;
            }
            if (!ok) {
                // let copies already in flight land before the CTA can exit
                mbar_drain(q_full, 0);
                for (int st = 0; st < NS; ++st) {
                    const int ck = nk > st ? (nk - 1 - st) / NS + 1 : 0;  // K loads issued to stage st
                    const int cv = nv > st ? (nv - 1 - st) / NS + 1 : 0;
                    if (ck > 0) mbar_drain(k_full + st, (ck - 1) & 1);
                    if (cv > 0) mbar_drain(v_full + st, (cv - 1) & 1);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0 && n_kv > 0) {
            constexpr uint32_t idS = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t idO = idesc_bf16(128, D, 0, 1);
            const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
            bool ok = mbar_wait(q_full, 0, ab, ROLE_MMA, 1);
            for (int it = 0; ok && it <= n_kv; ++it) {
                if (it < n_kv) {
                    const int st = it % NS;
                    if (!(ok = mbar_wait(k_full + st, (it / NS) & 1, ab, ROLE_MMA, 2))) break;
                    if (it > 0 && !(ok = mbar_wait(s_free, (it - 1) & 1, ab, ROLE_MMA, 3))) break;
                    tc_fence_after();
                    const uint32_t kbase = aK + st * C::TILE_BYTES;
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t off = (k >> 2) * C::CHUNK_BYTES + (k & 3) * 32;
                        umma_ss(tS, sdesc_sw128(aQ + off, 16, 1024), sdesc_sw128(kbase + off, 16, 1024), idS,
                                k > 0 ? 1u : 0u);
                    }
                    umma_commit(s_full);
                    umma_commit(k_empty + st);
                }
                if (it > 0) {
                    const int j = it - 1;
                    const int st = j % NS;
                    if (!(ok = mbar_wait(p_full, j & 1, ab, ROLE_MMA, 4))) break;
                    if (!(ok = mbar_wait(v_full + st, (j / NS) & 1, ab, ROLE_MMA, 5))) break;
                    tc_fence_after();
                    const uint32_t vbase = aV + st * C::TILE_BYTES;
#pragma unroll
                    for (int k = 0; k < kTile / 16; ++k)  // 16 keys = 8 TMEM columns of P per step
                        umma_ts(tO, tP + k * 8, sdesc_sw128(vbase + k * 2048, C::CHUNK_BYTES, 1024), idO,
                                (j > 0 || k > 0) ? 1u : 0u);
                    umma_commit(pv_done);
                    umma_commit(v_empty + st);
                }
            }
            if (!ok) {
                umma_commit(drain);
                mbar_drain(drain, 0);
            }
        }
    } else {
        // ------------------------------------------------------------------ softmax
        const int wq = warp & 3;                  // TMEM lane quadrant of this warp
        const int row = wq * 32 + lane;           // query row within the tile (TMEM lane)
        const uint32_t lane_off = uint32_t(wq * 32) << 16;
        const int s_row = qt * kTile + row;       // global query index
        float m_used = -INFINITY;                 // running max, log2 domain
        float l_sum = 0.f;
        bool ok = true;
        for (int it = 0; it < n_kv; ++it) {
            const int kt = fwd_kv_tile<MASK>(p, kv_first, it);
            ok = __all_sync(0xffffffffu, mbar_wait(s_full, it & 1, ab, ROLE_SOFTMAX, 1));
            if (!ok) break;
            tc_fence_after();
            float s[kTile];
#pragma unroll
            for (int c = 0; c < kTile / 32; ++c) tmem_ld32(tS + lane_off + c * 32, s + c * 32);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);

            const int k0 = kt * kTile;
            const bool diag = (MASK == ULYSSES_MASK_CAUSAL) && (kt == qt);
            const bool tail = k0 + kTile > p.L;
            if (diag || tail) {
#pragma unroll
                for (int c = 0; c < kTile; ++c) {
                    const int key = k0 + c;
                    if ((diag && key > s_row) || key >= p.L) s[c] = -INFINITY;
                }
            }
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < kTile; ++c) mx = fmaxf(mx, s[c]);
            const float m_new = fmaxf(m_used, mx * p.scale_log2);
            const bool need = m_new > m_used + 8.0f;
            if (it > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(pv_done, (it - 1) & 1, ab, ROLE_SOFTMAX, 2));
                if (!ok) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, need)) {
                    const float alpha = need ? ex2(m_used - m_new) : 1.0f;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        tmem_ld32(tO + lane_off + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        tmem_st32(tO + lane_off + c * 32, o);
                    }
                    tmem_wait_st();
                    l_sum *= alpha;
                }
            }
            if (need) m_used = m_new;
            const float neg_m = (m_used == -INFINITY) ? 0.f : -m_used;
            float rs = 0.f;
#pragma unroll
            for (int c = 0; c < kTile; ++c) {
                const float e = ex2(fmaf(s[c], p.scale_log2, neg_m));
                s[c] = e;
                rs += e;
            }
            l_sum += rs;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) pk[i] = pack_bf16(s[h2 * 64 + 2 * i], s[h2 * 64 + 2 * i + 1]);
                tmem_st32_u(tP + lane_off + h2 * 32, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }

        // ------------------------------------------------------------------ epilogue
        if (ok && n_kv > 0) ok = __all_sync(0xffffffffu, mbar_wait(pv_done, (n_kv - 1) & 1, ab, ROLE_EPI, 1));
        if (ok) {
            tc_fence_after();
            const bool valid = s_row < p.L;
            const bool any_key = l_sum > 0.f;
            const float inv_l = any_key ? 1.0f / l_sum : 0.f;
            __nv_bfloat16* orow;
            if (p.layout == ULYSSES_LAYOUT_TOKEN_SHARDED) {
                const int r = s_row / p.Lp, t = s_row % p.Lp;
                orow = static_cast<__nv_bfloat16*>(p.o) + ((size_t(r) * p.B + b) * p.Lp + t) * size_t(p.H) * D +
                       size_t(h) * D;
            } else {
                const int g = h / p.Hp, j = h % p.Hp;
                orow = static_cast<__nv_bfloat16*>(p.o) + ((size_t(g) * p.B + b) * p.L + s_row) * size_t(p.Hp) * D +
                       size_t(j) * D;
            }
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float o[32];
                if (n_kv > 0) {
                    tmem_ld32(tO + lane_off + c * 32, o);
                    tmem_wait_ld();
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = (n_kv > 0) ? o[i] * inv_l : 0.f;
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        dst[v] = make_uint4(pack_bf16(o[8 * v + 0], o[8 * v + 1]), pack_bf16(o[8 * v + 2], o[8 * v + 3]),
                                            pack_bf16(o[8 * v + 4], o[8 * v + 5]), pack_bf16(o[8 * v + 6], o[8 * v + 7]));
                    }
                }
            }
            if (valid) {
                const int g = h / p.Hp, j = h % p.Hp;
                const float lse = any_key ? (m_used + log2f(l_sum)) * 0.69314718055994531f : -INFINITY;
                p.lse[((size_t(g) * p.B + b) * p.Hp + j) * p.L + s_row] = lse;
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

template <int D, int MASK>
static int launch_fwd_t(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const FwdParams& p,
                        cudaStream_t stream) {
    using C = FwdCfg<D>;
    auto kern = attn_fwd_kernel<D, MASK>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_set[dev & 63]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
            return ULYSSES_ERR_CUDA;
        attr_set[dev & 63] = true;
    }
    dim3 grid(p.n_tiles, p.B * p.H);
    kern<<<grid, 192, C::SMEM_BYTES, stream>>>(mq, mk, mv, p);
    return cudaGetLastError() == cudaSuccess ? ULYSSES_OK : ULYSSES_ERR_CUDA;
}

int launch_attn_fwd(const ulysses_shape_t& s, const MaskArgs& m, float scale, int layout, const void* q,
                    const void* k, const void* v, void* o, float* lse, cudaStream_t stream) {
    FwdParams p{};
    p.B = s.B; p.L = s.L; p.H = s.H; p.P = s.P; p.Hp = s.H / s.P; p.Lp = s.L / s.P;
    p.layout = layout;
    p.n_tiles = (s.L + kTile - 1) / kTile;
    p.box_rows = layout == ULYSSES_LAYOUT_TOKEN_SHARDED ? gcd_int(p.Lp, kTile) : kTile;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.o = o;
    p.lse = lse;
    p.rowptr = m.q_rowptr;
    p.kcols = m.q_kcols;
    p.err = device_error_word();
    if (!p.err) return ULYSSES_ERR_CUDA;
    CUtensorMap mq, mk, mv;
    if (!encode_qkv_map(&mq, q, s, layout, p.box_rows) || !encode_qkv_map(&mk, k, s, layout, p.box_rows) ||
        !encode_qkv_map(&mv, v, s, layout, p.box_rows))
        return ULYSSES_ERR_CUDA;
    if (s.d_h == 128) {
        if (m.kind == ULYSSES_MASK_CAUSAL) return launch_fwd_t<128, ULYSSES_MASK_CAUSAL>(mq, mk, mv, p, stream);
        if (m.kind == ULYSSES_MASK_NONE) return launch_fwd_t<128, ULYSSES_MASK_NONE>(mq, mk, mv, p, stream);
        return launch_fwd_t<128, ULYSSES_MASK_BLOCK_SPARSE>(mq, mk, mv, p, stream);
    }
    if (m.kind == ULYSSES_MASK_CAUSAL) return launch_fwd_t<64, ULYSSES_MASK_CAUSAL>(mq, mk, mv, p, stream);
    if (m.kind == ULYSSES_MASK_NONE) return launch_fwd_t<64, ULYSSES_MASK_NONE>(mq, mk, mv, p, stream);
    return launch_fwd_t<64, ULYSSES_MASK_BLOCK_SPARSE>(mq, mk, mv, p, stream);
}

}  // namespace ulysses
