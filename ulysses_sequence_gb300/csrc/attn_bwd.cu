// Attention backward on the 5th-generation tensor cores: the analytic gradient of
// O = softmax(scale Q K^T + mask) V for one head over the full sequence (the pages leave
// the backward pass implicit in "training"; this is the textbook derivative):
//   P = exp(scale Q K^T - lse) on permitted pairs,  Delta_i = sum_e dO_ie O_ie,
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - Delta),  dQ = scale dS K,  dK = scale dS^T Q.
//
// Three kernels, all reading and writing through the token-sharded (or head-sharded)
// layout directly, so the backward relayouts (dO seq->head in, dQ/dK/dV head->seq out)
// are fused into the addressing:
//   1. bwd_prep:  Delta for every row (fp32) and a zeroed fp32 dQ accumulator;
//   2. attn_bwd_kernel: one CTA per (batch, head, 128-key tile), key/value stationary,
//      walking 64-row query steps. Per step, with S^T, dP^T in TMEM:
//        S^T  = K Q^T        (M=128 keys, N=64 queries, K=d)
//        dP^T = V dO^T       (M=128, N=64, K=d)
//        dV  += P^T dO       (M=128, N=d, K=64)     P^T bf16 in tensor memory (A operand)
//        dK  += dS^T Q       (M=128, N=d, K=64)     dS^T bf16 in tensor memory (A operand)
//        dQ^T = K^T dS^T     (M=d, N=64, K=128)     dS^T also in shared memory (B operand);
//                                                   added into the fp32 accumulator by
//                                                   bulk reductions from shared memory
//      Warps: 0 TMA producer (K, V once; Q, dO, lse, Delta per step, 3 stages), 1 MMA
//      issuer, 2-5 thread-per-key softmax/dS, 6-9 thread-per-feature dQ reduction.
//   3. bwd_dq_convert: dQ = bf16(scale * accumulator) into the output layout.
#include "common.cuh"
#include "ulysses_internal.h"

namespace ulysses {

struct BwdParams {
    int B, L, H, Hp, Lp, P;
    int layout;
    int n_ktiles;    // ceil(L / 128)
    int n_qsteps;    // ceil(L / 64)
    int box_rows_k;  // TMA box rows for 128-row key/value tiles
    int box_rows_q;  // TMA box rows for 64-row query steps
    float scale;
    float scale_log2;
    const float* lse;    // [P][B][Hp][L]
    const float* delta;  // [P][B][Hp][L]
    float* dq_acc;       // [B*H][n_qsteps][D/32][64][32]: one 8 KB block per (64 rows, 32 features)
    void* dk;
    void* dv;
    const int32_t* colptr;  // block-sparse CSC over key tiles
    const int32_t* qrows;
    uint32_t* err;
};

template <int D>
struct BwdCfg {
    static constexpr int NQ = 3;                            // query-step pipeline stages
    static constexpr uint32_t KT_BYTES = kTile * D * 2;     // 128-row key/value tile
    static constexpr uint32_t KCHUNK = kTile * 128;         // 128 rows x 64 elements
    static constexpr uint32_t QT_BYTES = kBwdQTile * D * 2; // 64-row query step
    static constexpr uint32_t QCHUNK = kBwdQTile * 128;     // 64 rows x 64 elements
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = OFF_K + KT_BYTES;
    static constexpr uint32_t OFF_Q = OFF_V + KT_BYTES;           // [NQ]
    static constexpr uint32_t OFF_DO = OFF_Q + NQ * QT_BYTES;     // [NQ]
    static constexpr uint32_t OFF_DST = OFF_DO + NQ * QT_BYTES;   // 128 x 64 bf16
    static constexpr uint32_t OFF_LSE = OFF_DST + kTile * kBwdQTile * 2;  // [NQ][64] fp32
    static constexpr uint32_t OFF_DELTA = OFF_LSE + NQ * kBwdQTile * 4;   // [NQ][64] fp32
    static constexpr int DQ_ROWS = 64;                                    // dQ rows staged per round
    static constexpr uint32_t OFF_DQS = OFF_DELTA + NQ * kBwdQTile * 4;   // [4 warps][DQ_ROWS][32] fp32
    static constexpr uint32_t DQS_WARP_BYTES = DQ_ROWS * 32 * 4;
    static constexpr uint32_t OFF_BAR = OFF_DQS + 4 * DQS_WARP_BYTES;
    static constexpr uint32_t SMEM_BYTES = OFF_BAR + 256 + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    // TMEM columns (P^T, dS^T: 64 bf16 per lane packed in 32 columns)
    static constexpr uint32_t T_S = 0, T_DP = 64, T_DQ = 128, T_PT = 192, T_DST = 224, T_DV = 256, T_DK = 384;
};

__device__ __forceinline__ void bwd_coords(const BwdParams& p, int s, int h, int& c1, int& c2, int& c4) {
    if (p.layout == ULYSSES_LAYOUT_TOKEN_SHARDED) {
        c1 = h;
        c2 = s % p.Lp;
        c4 = s / p.Lp;
    } else {
        c1 = h % p.Hp;
        c2 = s;
        c4 = h / p.Hp;
    }
}

// rows [s0, s0 + nrows) of head h into D/64 swizzled chunks of nrows x 64
template <int D>
__device__ __forceinline__ void bwd_load(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, const BwdParams& p,
                                         int s0, int nrows, int box_rows, int h, int b) {
    for (int c = 0; c < D / 64; ++c) {
        for (int r = 0; r < nrows; r += box_rows) {
            int c1, c2, c4;
            bwd_coords(p, s0 + r, h, c1, c2, c4);
            tma_load_5d(dst + c * nrows * 128 + r * 128, map, bar, c * 64, c1, c2, b, c4);
        }
    }
}

__device__ __forceinline__ size_t row_offset(const BwdParams& p, int s, int h, int b, int D) {
    if (p.layout == ULYSSES_LAYOUT_TOKEN_SHARDED) {
        const int r = s / p.Lp, t = s % p.Lp;
        return ((size_t(r) * p.B + b) * p.Lp + t) * size_t(p.H) * D + size_t(h) * D;
    }
    const int g = h / p.Hp, j = h % p.Hp;
    return ((size_t(g) * p.B + b) * p.L + s) * size_t(p.Hp) * D + size_t(j) * D;
}

__device__ __forceinline__ size_t stat_index(const BwdParams& p, int s, int h, int b) {
    const int g = h / p.Hp, j = h % p.Hp;
    return ((size_t(g) * p.B + b) * p.Hp + j) * p.L + s;
}

template <int MASK>
__device__ __forceinline__ int bwd_q_count(const BwdParams& p, int kt, int& first) {
    if (MASK == ULYSSES_MASK_CAUSAL) {
        first = 2 * kt;  // query steps before the key tile see none of its keys
        return p.n_qsteps - first;
    }
    if (MASK == ULYSSES_MASK_NONE) { first = 0; return p.n_qsteps; }
    first = p.colptr[kt];
    return 2 * (p.colptr[kt + 1] - first);
}

template <int MASK>
__device__ __forceinline__ int bwd_q_step(const BwdParams& p, int first, int it) {
    if (MASK == ULYSSES_MASK_BLOCK_SPARSE) return 2 * p.qrows[first + (it >> 1)] + (it & 1);
    return first + it;
}

template <int D, int MASK>
__global__ void __launch_bounds__(320, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const BwdParams p) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sK = smem + C::OFF_K;
    uint8_t* sV = smem + C::OFF_V;
    uint8_t* sQ = smem + C::OFF_Q;
    uint8_t* sDO = smem + C::OFF_DO;
    uint8_t* sDSt = smem + C::OFF_DST;
    float* sLSE = reinterpret_cast<float*>(smem + C::OFF_LSE);
    float* sDelta = reinterpret_cast<float*>(smem + C::OFF_DELTA);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    constexpr int NQ = C::NQ;
    uint64_t* kv_full = bars + 0;
    uint64_t* qdo_full = bars + 1;          // [NQ]
    uint64_t* qdo_empty = qdo_full + NQ;    // [NQ]
    uint64_t* s_full = qdo_empty + NQ;
    uint64_t* s_free = s_full + 1;
    uint64_t* dp_full = s_full + 2;
    uint64_t* dp_free = s_full + 3;
    uint64_t* p_full = s_full + 4;
    uint64_t* p_free = s_full + 5;
    uint64_t* ds_full = s_full + 6;
    uint64_t* ds_free = s_full + 7;
    uint64_t* dq_full = s_full + 8;
    uint64_t* dq_free = s_full + 9;
    uint64_t* dkdv_done = s_full + 10;
    uint64_t* drain = s_full + 11;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(s_full + 12);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = static_cast<int>(warp_id());
    const int lane = static_cast<int>(lane_id());
    // key tiles vary fastest, so the CTAs resident at one time share one head and its
    // fp32 dQ accumulator stays in L2
    const int bh = blockIdx.y;
    const int b = bh / p.H;
    const int h = bh % p.H;
    const int kt = blockIdx.x;
    int q_first = 0;
    const int n_it = bwd_q_count<MASK>(p, kt, q_first);

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        for (int i = 0; i < NQ; ++i) {
            mbar_init(qdo_full + i, 1);
            mbar_init(qdo_empty + i, 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_free, 4);
        mbar_init(dp_full, 1);
        mbar_init(dp_free, 4);
        mbar_init(p_full, 4);
        mbar_init(p_free, 1);
        mbar_init(ds_full, 4);
        mbar_init(ds_free, 1);
        mbar_init(dq_full, 1);
        mbar_init(dq_free, 4);
        mbar_init(dkdv_done, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Abort ab{abort_flag, p.err, KID_BWD};
    constexpr float kLog2e = 1.4426950408889634f;

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        bool ok = true;
        int nq = 0;
        if (n_it > 0) {
            if (lane == 0) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
                tma_prefetch_desc(&tm_do);
                mbar_arrive_expect_tx(kv_full, 2 * C::KT_BYTES);
                bwd_load<D>(sK, &tm_k, kv_full, p, kt * kTile, kTile, p.box_rows_k, h, b);
                bwd_load<D>(sV, &tm_v, kv_full, p, kt * kTile, kTile, p.box_rows_k, h, b);
            }
            // lse and Delta arrive by bulk copy when the 64-row step is whole and 16-byte aligned
            const bool bulk_stats = (p.L % 4) == 0;
            for (int it = 0; it < n_it; ++it) {
                const int st = it % NQ;
                if (it >= NQ) {
                    ok = __all_sync(0xffffffffu,
                                    mbar_wait(qdo_empty + st, ((it / NQ) - 1) & 1, ab, ROLE_LOAD, 1));
                    if (!ok) break;
                }
                const int q0 = bwd_q_step<MASK>(p, q_first, it) * kBwdQTile;
                const bool whole = bulk_stats && q0 + kBwdQTile <= p.L;
                if (!whole) {
                    for (int c = lane; c < kBwdQTile; c += 32) {
                        const int q = q0 + c;
                        const bool in = q < p.L;
                        sLSE[st * kBwdQTile + c] = in ? p.lse[stat_index(p, q, h, b)] : INFINITY;
                        sDelta[st * kBwdQTile + c] = in ? p.delta[stat_index(p, q, h, b)] : 0.f;
                    }
                    __syncwarp();
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(qdo_full + st, 2 * C::QT_BYTES + (whole ? 2 * kBwdQTile * 4 : 0));
                    if (whole) {
                        bulk_load(sLSE + st * kBwdQTile, p.lse + stat_index(p, q0, h, b), kBwdQTile * 4, qdo_full + st);
                        bulk_load(sDelta + st * kBwdQTile, p.delta + stat_index(p, q0, h, b), kBwdQTile * 4,
                                  qdo_full + st);
                    }
                    bwd_load<D>(sQ + st * C::QT_BYTES, &tm_q, qdo_full + st, p, q0, kBwdQTile, p.box_rows_q, h, b);
                    bwd_load<D>(sDO + st * C::QT_BYTES, &tm_do, qdo_full + st, p, q0, kBwdQTile, p.box_rows_q, h, b);
                }
                ++nq;
            }
            if (!ok && lane == 0) {
                mbar_drain(kv_full, 0);
                for (int st = 0; st < NQ; ++st) {
                    const int cnt = nq > st ? (nq - 1 - st) / NQ + 1 : 0;
                    if (cnt > 0) mbar_drain(qdo_full + st, (cnt - 1) & 1);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0 && n_it > 0) {
            constexpr uint32_t id_s = idesc_bf16(128, kBwdQTile, 0, 0);     // S^T, dP^T
            constexpr uint32_t id_kv = idesc_bf16(128, D, 0, 1);            // dV, dK
            constexpr uint32_t id_dq = idesc_bf16(128, kBwdQTile, 1, 1);    // dQ^T (M padded to 128 for d=64)
            const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aQ = smem_u32(sQ), aDO = smem_u32(sDO);
            const uint32_t aDSt = smem_u32(sDSt);
            const uint32_t tS = tmem + C::T_S, tDP = tmem + C::T_DP, tDQ = tmem + C::T_DQ;
            const uint32_t tDV = tmem + C::T_DV, tDK = tmem + C::T_DK;
            // K^T as an MN-major A operand: the second 64-row block of M is the second d chunk.
            // With d = 64 that block reads the V tile behind K; those lanes of dQ^T are ignored.
            const uint32_t kt_lbo = C::KCHUNK;

            // descriptors at the operands' base addresses; k-steps move them by constant offsets
            const uint64_t dK_k = sdesc_sw128(aK, 16, 1024), dV_k = sdesc_sw128(aV, 16, 1024);
            const uint64_t dKt_mn = sdesc_sw128(aK, kt_lbo, 1024), dDSt_mn = sdesc_sw128(aDSt, C::QCHUNK, 1024);
            auto issue_s_dp = [&](int j) {
                const int st = j % NQ;
                const uint64_t dQ_k = sdesc_sw128(aQ + st * C::QT_BYTES, 16, 1024);
                const uint64_t dDO_k = sdesc_sw128(aDO + st * C::QT_BYTES, 16, 1024);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t ko = (k >> 2) * C::KCHUNK + (k & 3) * 32;
                    const uint32_t qo = (k >> 2) * C::QCHUNK + (k & 3) * 32;
                    umma_ss(tS, sdesc_add(dK_k, ko), sdesc_add(dQ_k, qo), id_s, k > 0);
                }
                umma_commit(s_full);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t ko = (k >> 2) * C::KCHUNK + (k & 3) * 32;
                    const uint32_t qo = (k >> 2) * C::QCHUNK + (k & 3) * 32;
                    umma_ss(tDP, sdesc_add(dV_k, ko), sdesc_add(dDO_k, qo), id_s, k > 0);
                }
                umma_commit(dp_full);
            };

            bool ok = mbar_wait(kv_full, 0, ab, ROLE_MMA, 1) && mbar_wait(qdo_full, 0, ab, ROLE_MMA, 2);
            if (ok) {
                tc_fence_after();
                issue_s_dp(0);
            }
            for (int it = 0; ok && it < n_it; ++it) {
                const int st = it % NQ;
                const uint64_t dQ_mn = sdesc_sw128(aQ + st * C::QT_BYTES, C::QCHUNK, 1024);
                const uint64_t dDO_mn = sdesc_sw128(aDO + st * C::QT_BYTES, C::QCHUNK, 1024);
                // dV += P^T dO
                if (!(ok = mbar_wait(p_full, it & 1, ab, ROLE_MMA, 3))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < kBwdQTile / 16; ++k)  // 16 queries = 8 TMEM columns of P^T
                    umma_ts(tDV, tmem + C::T_PT + k * 8, sdesc_add(dDO_mn, k * 2048), id_kv, (it > 0 || k > 0) ? 1u : 0u);
                umma_commit(p_free);
                // next step's S^T and dP^T overlap this step's dS computation
                if (it + 1 < n_it) {
                    if (!(ok = mbar_wait(qdo_full + ((it + 1) % NQ), ((it + 1) / NQ) & 1, ab, ROLE_MMA, 4))) break;
                    if (!(ok = mbar_wait(s_free, it & 1, ab, ROLE_MMA, 5))) break;
                    if (!(ok = mbar_wait(dp_free, it & 1, ab, ROLE_MMA, 6))) break;
                    tc_fence_after();
                    issue_s_dp(it + 1);
                }
                // dK += dS^T Q ;  dQ^T = K^T dS^T
                if (!(ok = mbar_wait(ds_full, it & 1, ab, ROLE_MMA, 7))) break;
                if (it > 0 && !(ok = mbar_wait(dq_free, (it - 1) & 1, ab, ROLE_MMA, 8))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < kBwdQTile / 16; ++k)  // 16 queries = 8 TMEM columns of dS^T
                    umma_ts(tDK, tmem + C::T_DST + k * 8, sdesc_add(dQ_mn, k * 2048), id_kv, (it > 0 || k > 0) ? 1u : 0u);
#pragma unroll
                for (int k = 0; k < kTile / 16; ++k)
                    umma_ss(tDQ, sdesc_add(dKt_mn, k * 2048), sdesc_add(dDSt_mn, k * 2048), id_dq, k > 0 ? 1u : 0u);
                umma_commit(dq_full);
                umma_commit(ds_free);
                umma_commit(qdo_empty + st);
            }
            if (ok) umma_commit(dkdv_done);
            else {
                umma_commit(drain);
                mbar_drain(drain, 0);
            }
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------------ softmax / dS
        const int wq = warp & 3;
        const int row = wq * 32 + lane;  // key row within the tile (TMEM lane)
        const uint32_t lane_off = uint32_t(wq * 32) << 16;
        const int key = kt * kTile + row;
        const uint32_t aDSt = smem_u32(sDSt);
        bool ok = true;
        for (int it = 0; it < n_it; ++it) {
            const int st = it % NQ;
            const int q0 = bwd_q_step<MASK>(p, q_first, it) * kBwdQTile;
            ok = __all_sync(0xffffffffu, mbar_wait(qdo_full + st, (it / NQ) & 1, ab, ROLE_SOFTMAX, 1) &&
                                             mbar_wait(s_full, it & 1, ab, ROLE_SOFTMAX, 2));
            if (!ok) break;
            tc_fence_after();
            float pv[kBwdQTile];
            tmem_ld32(tmem + C::T_S + lane_off, pv);
            tmem_ld32(tmem + C::T_S + lane_off + 32, pv + 32);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);
            const float* lse = sLSE + st * kBwdQTile;
            const bool diag = (MASK == ULYSSES_MASK_CAUSAL) && (q0 < kt * kTile + kTile);
#pragma unroll
            for (int c = 0; c < kBwdQTile; ++c) {
                float e = ex2(fmaf(pv[c], p.scale_log2, -lse[c] * kLog2e));
                if (diag && q0 + c < key) e = 0.f;
                pv[c] = e;
            }
            if (it > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(p_free, (it - 1) & 1, ab, ROLE_SOFTMAX, 3));
                if (!ok) break;
            }
            {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) pk[i] = pack_bf16(pv[2 * i], pv[2 * i + 1]);
                tmem_st32_u(tmem + C::T_PT + lane_off, pk);
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);

            ok = __all_sync(0xffffffffu, mbar_wait(dp_full, it & 1, ab, ROLE_SOFTMAX, 4));
            if (!ok) break;
            tc_fence_after();
            float dp[kBwdQTile];
            tmem_ld32(tmem + C::T_DP + lane_off, dp);
            tmem_ld32(tmem + C::T_DP + lane_off + 32, dp + 32);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dp_free);
            const float* dl = sDelta + st * kBwdQTile;
#pragma unroll
            for (int c = 0; c < kBwdQTile; ++c) dp[c] = pv[c] * (dp[c] - dl[c]);
            if (it > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(ds_free, (it - 1) & 1, ab, ROLE_SOFTMAX, 5));
                if (!ok) break;
            }
            {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) pk[i] = pack_bf16(dp[2 * i], dp[2 * i + 1]);
                tmem_st32_u(tmem + C::T_DST + lane_off, pk);  // A operand of dK
#pragma unroll
                for (int u = 0; u < 8; ++u)                    // B operand of dQ^T
                    st_shared_v4(aDSt + sw128_offset(row, u), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(ds_full);
        }
        // ------------------------------------------------------------------ dK, dV epilogue
        if (ok && n_it > 0) ok = __all_sync(0xffffffffu, mbar_wait(dkdv_done, 0, ab, ROLE_EPI, 1));
        if (ok) {
            tc_fence_after();
            const bool valid = key < p.L;
            const size_t off = row_offset(p, key, h, b, D);
            for (int which = 0; which < 2; ++which) {
                const uint32_t tcol = which == 0 ? C::T_DV : C::T_DK;
                const float mul = which == 0 ? 1.0f : p.scale;
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(which == 0 ? p.dv : p.dk) + off;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float v[32];
                    if (n_it > 0) {
                        tmem_ld32(tmem + tcol + lane_off + c * 32, v);
                        tmem_wait_ld();
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = (n_it > 0) ? v[i] * mul : 0.f;
                    if (valid) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                        for (int x = 0; x < 4; ++x)
                            d4[x] = make_uint4(pack_bf16(v[8 * x], v[8 * x + 1]), pack_bf16(v[8 * x + 2], v[8 * x + 3]),
                                               pack_bf16(v[8 * x + 4], v[8 * x + 5]),
                                               pack_bf16(v[8 * x + 6], v[8 * x + 7]));
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------------ dQ reduction
        // Thread e holds dQ^T[e][0..63] of this step. Each warp stages its 32 features x 64
        // rows in shared memory ([row][32] fp32, one 128-byte line per row) and adds the 8 KB
        // block to the accumulator with one bulk reduction performed at L2. (Staging in
        // smaller rounds, to free room for a fourth query stage, measured slower.)
        const int wq = warp & 3;
        const int e = wq * 32 + lane;  // feature index (TMEM lane of dQ^T)
        const uint32_t lane_off = uint32_t(wq * 32) << 16;
        const uint32_t stage = smem_u32(smem + C::OFF_DQS + wq * C::DQS_WARP_BYTES);
        float* acc_head = p.dq_acc + size_t(b * p.H + h) * p.n_qsteps * kBwdQTile * D;
        bool pending = false;
        for (int it = 0; it < n_it; ++it) {
            const int qs = bwd_q_step<MASK>(p, q_first, it);
            if (!__all_sync(0xffffffffu, mbar_wait(dq_full, it & 1, ab, ROLE_DQ, 1))) break;
            tc_fence_after();
            float v[kBwdQTile];
            tmem_ld32(tmem + C::T_DQ + lane_off, v);
            tmem_ld32(tmem + C::T_DQ + lane_off + 32, v + 32);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dq_free);
            if (e < D) {  // warp-uniform: d = 64 leaves the upper two warps idle
                float* block = acc_head + (size_t(qs) * (D / 32) + wq) * (kBwdQTile * 32);
#pragma unroll
                for (int r0 = 0; r0 < kBwdQTile; r0 += C::DQ_ROWS) {
                    if (pending) {
                        if (lane == 0) bulk_wait_read_all();  // the previous piece has left the stage
                        __syncwarp();
                    }
#pragma unroll
                    for (int c = 0; c < C::DQ_ROWS; ++c) st_shared_f32(stage + c * 128 + lane * 4, v[r0 + c]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        bulk_reduce_add_f32(block + r0 * 32, smem + C::OFF_DQS + wq * C::DQS_WARP_BYTES,
                                            C::DQS_WARP_BYTES);
                        bulk_commit();
                    }
                    pending = true;
                }
            }
        }
        if (pending && lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncwarp();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// Delta_i = sum_e dO_ie O_ie (fp32) for every row, and the fp32 dQ accumulator set to 0.
// Eight lanes per row, each with one 16-byte vector of O and dO per 64 features.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(BwdParams p, const __nv_bfloat16* o, const __nv_bfloat16* dO,
                                                       float* delta) {
    constexpr int LPR = 8;              // lanes per row
    constexpr int VPT = D / (8 * LPR);  // 16-byte vectors per lane
    const size_t rows = size_t(p.B) * p.H * p.L;
    const int sub = threadIdx.x % LPR;
    const size_t gwarp = (size_t(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
    const size_t nwarps = size_t(gridDim.x) * blockDim.x / 32;
    // every lane of a warp runs the same number of iterations (the shuffle needs all 32)
    for (size_t base = gwarp * 4; base < rows; base += nwarps * 4) {
        const size_t rr = base + (threadIdx.x % 32) / LPR;  // rows enumerated as (b, h, s)
        const bool in = rr < rows;
        float sum = 0.f;
        int s = 0, h = 0, b = 0;
        if (in) {
            s = int(rr % p.L);
            const size_t bh = rr / p.L;
            h = int(bh % p.H);
            b = int(bh / p.H);
            const size_t off = row_offset(p, s, h, b, D);
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int e0 = (sub + v * LPR) * 8;
                const uint4 a = *reinterpret_cast<const uint4*>(o + off + e0);
                const uint4 g = *reinterpret_cast<const uint4*>(dO + off + e0);
                const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
                const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 af = __bfloat1622float2(a2[i]);
                    const float2 gf = __bfloat1622float2(g2[i]);
                    sum = fmaf(af.x, gf.x, sum);
                    sum = fmaf(af.y, gf.y, sum);
                }
            }
        }
#pragma unroll
        for (int m = LPR / 2; m > 0; m >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, m);
        if (in && sub == 0) delta[stat_index(p, s, h, b)] = sum;
    }
    // zero the fp32 dQ accumulator (tile layout, padded to whole 64-row steps)
    const size_t n4 = size_t(p.B) * p.H * p.n_qsteps * kBwdQTile * D / 4;
    float4* acc = reinterpret_cast<float4*>(p.dq_acc);
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += size_t(gridDim.x) * blockDim.x)
        acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// dQ = bf16(scale * accumulator), written in the output layout.
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(BwdParams p, __nv_bfloat16* dq) {
    constexpr int LPR = 8;
    constexpr int VPT = D / (8 * LPR);
    const size_t rows = size_t(p.B) * p.H * p.L;
    const int sub = threadIdx.x % LPR;
    for (size_t rr = (size_t(blockIdx.x) * blockDim.x + threadIdx.x) / LPR; rr < rows;
         rr += size_t(gridDim.x) * blockDim.x / LPR) {
        const int s = int(rr % p.L);
        const size_t bh = rr / p.L;
        const int h = int(bh % p.H);
        const int b = int(bh / p.H);
        const size_t off = row_offset(p, s, h, b, D);
        // tile layout [b*H + h][s / 64][e / 32][s % 64][e % 32]
        const float* acc = p.dq_acc + (bh * p.n_qsteps + s / kBwdQTile) * size_t(kBwdQTile) * D + (s % kBwdQTile) * 32;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int e0 = (sub + v * LPR) * 8;
            const float* a = acc + (e0 / 32) * (kBwdQTile * 32) + (e0 % 32);
            const float4 x0 = *reinterpret_cast<const float4*>(a);
            const float4 x1 = *reinterpret_cast<const float4*>(a + 4);
            *reinterpret_cast<uint4*>(dq + off + e0) =
                make_uint4(pack_bf16(x0.x * p.scale, x0.y * p.scale), pack_bf16(x0.z * p.scale, x0.w * p.scale),
                           pack_bf16(x1.x * p.scale, x1.y * p.scale), pack_bf16(x1.z * p.scale, x1.w * p.scale));
        }
    }
}

static size_t acc_bytes(const ulysses_shape_t& s) {
    const size_t steps = (size_t(s.L) + kBwdQTile - 1) / kBwdQTile;
    return (size_t(s.B) * s.H * steps * kBwdQTile * s.d_h * 4 + 255) / 256 * 256;
}

size_t bwd_workspace_bytes(const ulysses_shape_t& s) {
    const size_t rows = size_t(s.B) * s.H * s.L;
    return acc_bytes(s) + (rows * 4 + 255) / 256 * 256;
}

template <int D, int MASK>
static int launch_bwd_t(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdo,
                        const BwdParams& p, cudaStream_t stream) {
    using C = BwdCfg<D>;
    auto kern = attn_bwd_kernel<D, MASK>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (!attr_set[dev & 63]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
            return ULYSSES_ERR_CUDA;
        attr_set[dev & 63] = true;
    }
    dim3 grid(p.n_ktiles, p.B * p.H);
    kern<<<grid, 320, C::SMEM_BYTES, stream>>>(mq, mk, mv, mdo, p);
    return cudaGetLastError() == cudaSuccess ? ULYSSES_OK : ULYSSES_ERR_CUDA;
}

template <int D>
static int launch_bwd_d(const ulysses_shape_t& s, const MaskArgs& m, BwdParams& p, const void* q, const void* k,
                        const void* v, const void* o, const void* dO, void* dq, cudaStream_t stream) {
    CUtensorMap mq, mk, mv, mdo;
    if (!encode_qkv_map(&mq, q, s, p.layout, p.box_rows_q) || !encode_qkv_map(&mdo, dO, s, p.layout, p.box_rows_q) ||
        !encode_qkv_map(&mk, k, s, p.layout, p.box_rows_k) || !encode_qkv_map(&mv, v, s, p.layout, p.box_rows_k))
        return ULYSSES_ERR_CUDA;
    const int sms = device_sm_count();
    const size_t rows = size_t(s.B) * s.H * s.L;
    size_t blocks = (rows * 8 + 255) / 256;
    if (blocks > size_t(sms) * 16) blocks = size_t(sms) * 16;
    bwd_prep_kernel<D><<<unsigned(blocks), 256, 0, stream>>>(p, static_cast<const __nv_bfloat16*>(o),
                                                              static_cast<const __nv_bfloat16*>(dO),
                                                              const_cast<float*>(p.delta));
    if (cudaGetLastError() != cudaSuccess) return ULYSSES_ERR_CUDA;
    int rc;
    if (m.kind == ULYSSES_MASK_CAUSAL) rc = launch_bwd_t<D, ULYSSES_MASK_CAUSAL>(mq, mk, mv, mdo, p, stream);
    else if (m.kind == ULYSSES_MASK_NONE) rc = launch_bwd_t<D, ULYSSES_MASK_NONE>(mq, mk, mv, mdo, p, stream);
    else rc = launch_bwd_t<D, ULYSSES_MASK_BLOCK_SPARSE>(mq, mk, mv, mdo, p, stream);
    if (rc != ULYSSES_OK) return rc;
    bwd_dq_convert_kernel<D><<<unsigned(blocks), 256, 0, stream>>>(p, static_cast<__nv_bfloat16*>(dq));
    return cudaGetLastError() == cudaSuccess ? ULYSSES_OK : ULYSSES_ERR_CUDA;
}

int launch_attn_bwd(const ulysses_shape_t& s, const MaskArgs& m, float scale, int layout, const void* q,
                    const void* k, const void* v, const void* o, const float* lse, const void* dO, void* dq,
                    void* dk, void* dv, void* workspace, cudaStream_t stream) {
    BwdParams p{};
    p.B = s.B; p.L = s.L; p.H = s.H; p.P = s.P; p.Hp = s.H / s.P; p.Lp = s.L / s.P;
    p.layout = layout;
    p.n_ktiles = (s.L + kTile - 1) / kTile;
    p.n_qsteps = (s.L + kBwdQTile - 1) / kBwdQTile;
    p.box_rows_k = layout == ULYSSES_LAYOUT_TOKEN_SHARDED ? gcd_int(p.Lp, kTile) : kTile;
    p.box_rows_q = layout == ULYSSES_LAYOUT_TOKEN_SHARDED ? gcd_int(p.Lp, kBwdQTile) : kBwdQTile;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.lse = lse;
    p.dq_acc = static_cast<float*>(workspace);
    p.delta = reinterpret_cast<float*>(static_cast<char*>(workspace) + acc_bytes(s));
    p.dk = dk;
    p.dv = dv;
    p.colptr = m.k_colptr;
    p.qrows = m.k_qrows;
    p.err = device_error_word();
    if (!p.err) return ULYSSES_ERR_CUDA;
    if (s.d_h == 128) return launch_bwd_d<128>(s, m, p, q, k, v, o, dO, dq, stream);
    return launch_bwd_d<64>(s, m, p, q, k, v, o, dO, dq, stream);
}

}  // namespace ulysses
