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
//      walking 128-row query steps. Every MMA is 128 x 128 (narrower MMAs take nearly as
//      long on the tensor cores, so they would waste half of it):
//        S^T  = K Q^T     (M=128 keys, N=128 queries, K=d)    -> TMEM columns [0, 128)
//        dP^T = V dO^T    (M=128, N=128, K=d)                  -> TMEM columns [128, 256)
//        dV  += P^T dO    (M=128, N=d, K=128)   P^T bf16 in tensor memory over S^T
//        dQ^T = K^T dS^T  (M=d, N=128, K=128)   dS^T bf16 in shared memory (B operand),
//                                               written over dP^T once the softmax warps have
//                                               read it, then added into the fp32 accumulator
//                                               by bulk reductions
//        dK  += dS^T Q    (M=128, N=d, K=128)   the same dS^T buffer as a K-major A operand
//      The next step's S^T is issued right after dV, so the exponentials of the next P
//      overlap dQ^T and dK on the tensor cores; dQ^T goes before dK, so the drain warps read
//      it out of tensor memory while dK runs and the next dP^T can follow dK at once.
//      Warps: 0 TMA producer (K, V once; per step Q into one of two slots, dO into one),
//      1 MMA issuer, 2-9 softmax and dS, two warps per tensor-memory lane quadrant, each
//      taking 64 of the step's 128 queries, 10-13 dQ drain, one per lane quadrant (and one
//      per SM sub-partition): each reads its 32 features x 128 queries of dQ^T out of tensor
//      memory and issues every reduction, so none of them sits in the softmax warps' loop.
//      Fourteen warps leave 144 registers per thread.
//   3. bwd_dq_convert: dQ = bf16(scale * accumulator) into the output layout.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "ulysses_internal.h"

namespace ulysses {

constexpr int kQStep = 128;  // query rows per step of the backward kernel
constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
    int B, L, H, Hp, Lp, P;
    int Hkv, G, Hkvp, kv_rep;  // key/value heads, query heads per key/value head, per group, copies
    int layout;
    int n_tiles;     // ceil(L / 128): key tiles and query steps
    int box_rows;    // TMA box rows (divides 128; boxes never straddle a shard)
    float scale;
    float scale_log2;
    const float* lse;    // [P][B][Hp][L]
    const float* delta;  // [P][B][Hp][L]
    float* dq_acc;       // fp32 dQ^T blocks (dq_block), rows past L padding
    void* dk;
    void* dv;
    const int32_t* colptr;  // block-sparse CSC over key tiles
    const int32_t* qrows;
    uint32_t* err;
};

// The accumulating kernels' parameters (a separate type: growing BwdParams itself measurably
// slowed the plain kernel)
struct BwdAccParams : BwdParams {
    float* dk_acc;   // fp32 accumulators of dK, dV (layout of dK)
    float* dv_acc;
    int dkv_mode;    // 1 fp32 store, 2 fp32 add, 3 bf16(accumulator + part)
};
template <bool ACC>
using BwdParamsOf = typename std::conditional<ACC, BwdAccParams, BwdParams>::type;

template <int D>
struct BwdCfg {
    static constexpr uint32_t T_BYTES = kTile * D * 2;   // 128-row tile (K, V, Q or dO)
    static constexpr uint32_t CHUNK = kTile * 128;       // 128 rows x 64 elements
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = OFF_K + T_BYTES;
    static constexpr uint32_t OFF_Q = OFF_V + T_BYTES;     // [2] slots
    static constexpr uint32_t OFF_DO = OFF_Q + 2 * T_BYTES;
    static constexpr uint32_t OFF_DST = OFF_DO + T_BYTES;  // dS^T: 2 chunks of 128 keys x 64 queries
    static constexpr uint32_t DST_BYTES = kTile * kQStep * 2;
    static constexpr uint32_t OFF_LSE = OFF_DST + DST_BYTES;    // [2][128] fp32
    static constexpr uint32_t OFF_DELTA = OFF_LSE + 2 * kQStep * 4;  // [2][128] fp32
    // each drain warp's private staging of 64 of its dQ^T columns: 32 lanes x 64 fp32 (8 KB)
    static constexpr uint32_t OFF_STG = OFF_DELTA + 2 * kQStep * 4;
    static constexpr uint32_t STG_BYTES = 4 * 8192;
    static constexpr uint32_t OFF_BAR = OFF_STG + STG_BYTES;
    // 1 KB of slack to align the dynamic shared memory base where it fits; without it the
    // kernel checks that the base is 1024-byte aligned (it is, after the 1 KB the system keeps)
    static constexpr uint32_t SLACK = OFF_BAR + 256 + 1024 <= 232448 ? 1024 : 0;
    static constexpr uint32_t SMEM_BYTES = OFF_BAR + 256 + SLACK;
    static constexpr uint32_t TMEM_COLS = 512;
    // tensor-memory columns: S^T (then P^T), dP^T (then dQ^T), dV, dK
    static constexpr uint32_t T_S = 0, T_DP = 128, T_DV = 256, T_DK = 256 + D;
    static_assert(T_DK + D <= TMEM_COLS, "tensor memory");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

__device__ __forceinline__ void bwd_coords(const BwdParams& p, int s, int h, int& c1, int& c2, int& c4) {
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

// rows [s0, s0 + 128) of head h into D/64 swizzled chunks of 128 x 64
template <int D>
__device__ __forceinline__ void bwd_load(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, const BwdParams& p,
                                         int s0, int h, int b) {
    for (int c = 0; c < D / 64; ++c) {
        for (int r = 0; r < kTile; r += p.box_rows) {
            int c1, c2, c4;
            bwd_coords(p, s0 + r, h, c1, c2, c4);
            tma_load_5d(dst + c * BwdCfg<D>::CHUNK + r * 128, map, bar, c * 64, c1, c2, b, c4);
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

// The key/value head a CTA of the backward owns (grid y = unit), and the query heads that
// attend with it: h_first .. h_first + nqh - 1.
struct KvUnit {
    int b;
    int kv;       // key/value head: in the token layout its index, in the head layout its index within group g
    int g;        // head group (head layout)
    int h_first;  // first query head
    int nqh;      // query heads
};

__device__ __forceinline__ KvUnit kv_unit(const BwdParams& p, int unit) {
    KvUnit u;
    if (p.layout == ULYSSES_LAYOUT_TOKEN_SHARDED) {
        u.b = unit / p.Hkv;
        u.kv = unit % p.Hkv;
        u.g = 0;
        u.h_first = u.kv * p.G;
        u.nqh = p.G;
    } else {
        u.g = unit / (p.B * p.Hkvp);
        const int rem = unit % (p.B * p.Hkvp);
        u.b = rem / p.Hkvp;
        u.kv = rem % p.Hkvp;
        // without copies the group's query heads split into Hkvp runs of G; with copies every
        // query head of the group attends with the group's one key/value head
        u.h_first = u.g * p.Hp + (p.kv_rep == 1 ? u.kv * p.G : 0);
        u.nqh = p.kv_rep == 1 ? p.G : p.Hp;
    }
    return u;
}

// K/V coordinates of global row s for the unit's key/value head
__device__ __forceinline__ void kv_coords(const BwdParams& p, int s, const KvUnit& u, int& c1, int& c2, int& c4) {
    c1 = u.kv;
    if (p.layout == ULYSSES_LAYOUT_TOKEN_SHARDED) {
        c2 = s % p.Lp;
        c4 = s / p.Lp;
    } else {
        c2 = s;
        c4 = u.g;
    }
}

// rows [s0, s0 + 128) of the unit's key/value head into D/64 swizzled chunks of 128 x 64
template <int D>
__device__ __forceinline__ void kv_load(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, const BwdParams& p,
                                        int s0, const KvUnit& u) {
    for (int c = 0; c < D / 64; ++c) {
        for (int r = 0; r < kTile; r += p.box_rows) {
            int c1, c2, c4;
            kv_coords(p, s0 + r, u, c1, c2, c4);
            tma_load_5d(dst + c * BwdCfg<D>::CHUNK + r * 128, map, bar, c * 64, c1, c2, u.b, c4);
        }
    }
}

// element offset of row s of the unit's key/value head in a K/V-shaped tensor
__device__ __forceinline__ size_t kv_row_offset(const BwdParams& p, int s, const KvUnit& u, int D) {
    if (p.layout == ULYSSES_LAYOUT_TOKEN_SHARDED) {
        const int r = s / p.Lp, t = s % p.Lp;
        return ((size_t(r) * p.B + u.b) * p.Lp + t) * size_t(p.Hkv) * D + size_t(u.kv) * D;
    }
    return ((size_t(u.g) * p.B + u.b) * p.L + s) * size_t(p.Hkvp) * D + size_t(u.kv) * D;
}

__device__ __forceinline__ size_t stat_index(const BwdParams& p, int s, int h, int b) {
    const int g = h / p.Hp, j = h % p.Hp;
    return ((size_t(g) * p.B + b) * p.Hp + j) * p.L + s;
}

// The fp32 dQ accumulator is a sequence of 8 KB blocks, one per (batch x head, query step,
// query half hq, feature quadrant wq): 32 features x 64 queries of dQ^T, the rows one drain
// warp reads out of tensor memory. Feature lane l holds its 64 queries as 16 units of four
// floats, unit u at position u ^ (l & 7), so that the eight lanes of each 128-byte access
// phase of the warp's 16-byte stores hit different bank groups. A block is added into
// global memory as it lies in shared memory, by one bulk reduction.
constexpr uint32_t kDqBlockFloats = 32 * 64;
template <int D>
__device__ __forceinline__ size_t dq_block(const BwdParams& p, int bh, int qstep, int hq, int wq) {
    return ((size_t(bh) * p.n_tiles + qstep) * 2 + hq) * size_t(D / 32) + wq;
}

// The block-sparse schedule, four arrays of n_tiles ints in the workspace behind Delta:
// order (key tiles by descending CSC length, ties by index), their lengths, and for each
// position of order the start and size of its class (the run of equal lengths).
__device__ __forceinline__ const int32_t* bwd_schedule(const BwdParams& p) {
    const size_t rows = size_t(p.B) * p.H * p.L;
    return reinterpret_cast<const int32_t*>(p.delta + (rows + 63) / 64 * 64);
}

// The key tile and key/value unit of this CTA. Block-sparse masks deal the CTAs out longest
// first: tiles of one length class go out together, unit by unit within the class, so that the
// long tiles (a global key tile walks every query tile) start in the first waves, and the
// long tiles of one (batch, head) run side by side and share its Q and dO in L2.
template <int MASK>
__device__ __forceinline__ void bwd_cta_tile(const BwdParams& p, int units, int& kt, int& unit) {
    if (MASK != ULYSSES_MASK_BLOCK_SPARSE) {
        kt = blockIdx.x;
        unit = blockIdx.y;
        return;
    }
    const int32_t* sched = bwd_schedule(p);
    const int n = p.n_tiles;
    const int64_t i = int64_t(blockIdx.y) * n + blockIdx.x;
    const int pos = int(i / units);
    const int start = sched[2 * n + pos], size = sched[3 * n + pos];
    const int64_t j = i - int64_t(start) * units;
    unit = int(j / size);
    kt = sched[start + int(j % size)];
}

// Causal grids with short sequences deal out groups of G units (G = gridDim.x / n_tiles,
// chosen so that their Q, dO and dQ accumulator fit in a quarter of L2), longest key tile
// first across the group, so that the light tiles of every unit fill the last waves. Returns
// false for the last group's spare CTAs, which have no tile.
__device__ __forceinline__ bool bwd_cta_tile_grouped(const BwdParams& p, int& kt, int& unit) {
    const int all = p.layout == ULYSSES_LAYOUT_TOKEN_SHARDED ? p.B * p.Hkv : p.P * p.B * p.Hkvp;
    const int G = int(gridDim.x) / p.n_tiles;
    const int Gg = min(G, all - int(blockIdx.y) * G);
    const int r = int(blockIdx.x);
    if (r >= Gg * p.n_tiles) return false;
    kt = r / Gg;
    unit = int(blockIdx.y) * G + r % Gg;
    return true;
}

template <int MASK>
__device__ __forceinline__ int bwd_q_count(const BwdParams& p, int kt, int& first) {
    if (MASK == ULYSSES_MASK_CAUSAL) {
        first = kt;  // query steps before the key tile see none of its keys
        return p.n_tiles - kt;
    }
    if (MASK == ULYSSES_MASK_NONE) { first = 0; return p.n_tiles; }
    first = p.colptr[kt];
    return p.colptr[kt + 1] - first;
}

template <int MASK>
__device__ __forceinline__ int bwd_q_step(const BwdParams& p, int first, int it) {
    if (MASK == ULYSSES_MASK_BLOCK_SPARSE) return p.qrows[first + it];
    return first + it;
}

// Two warps share each tensor-memory lane quadrant; warp half hf takes queries
// [64 hf, 64 hf + 64) of a step and writes its 64 bf16 results (32 packed columns) inside
// the 64 columns it read itself: half 0 at [0, 32), half 1 at [96, 128). The K-step k (16
// queries) of an MMA reading them as its A operand therefore starts at column a_col(k).
__device__ __forceinline__ uint32_t a_col(int k) { return uint32_t(8 * k + (k >= 4 ? 64 : 0)); }

// ACC: dK, dV go through the fp32 accumulators (dkv_mode 1-3) instead of straight to bf16
// Warps of the backward kernel: producer, MMA issuer, 8 softmax, 4 dQ drain
constexpr int kBwdThreads = 14 * 32;

template <int D, int MASK, bool ACC, bool GRP = false>
__global__ void __launch_bounds__(kBwdThreads, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const BwdParamsOf<ACC> p) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    if (C::SLACK == 0 && (smem_u32(smem_raw) & 1023u) != 0) {
        // uniform early exit, before any barrier or tensor memory exists
        if (threadIdx.x == 0) record_error(p.err, (KID_BWD << 24) | (ROLE_LOAD << 16) | 0xa1u);
        return;
    }
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sK = smem + C::OFF_K;
    uint8_t* sV = smem + C::OFF_V;
    uint8_t* sQ = smem + C::OFF_Q;
    uint8_t* sDO = smem + C::OFF_DO;
    uint8_t* sDSt = smem + C::OFF_DST;
    float* sLSE = reinterpret_cast<float*>(smem + C::OFF_LSE);
    float* sDelta = reinterpret_cast<float*>(smem + C::OFF_DELTA);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* kv_full = bars + 0;
    uint64_t* q_full = bars + 1;      // [2] Q slot + its lse, Delta
    uint64_t* q_empty = bars + 3;     // [2]
    uint64_t* do_full = bars + 5;
    uint64_t* do_empty = bars + 6;
    uint64_t* s_full = bars + 7;
    uint64_t* dp_full = bars + 8;
    uint64_t* p_full = bars + 9;      // 8 warps
    uint64_t* ds_full = bars + 10;    // 8 warps
    uint64_t* dq_full = bars + 11;
    uint64_t* dq_free = bars + 12;    // 4 drain warps
    uint64_t* dkdv_done = bars + 13;
    uint64_t* drain = bars + 14;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 15);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = static_cast<int>(warp_id());
    const int lane = static_cast<int>(lane_id());
    // key tiles vary fastest, so the CTAs resident at one time share one head and its
    // fp32 dQ accumulator stays in L2
    int kt, unit;
    if constexpr (GRP) {
        if (!bwd_cta_tile_grouped(p, kt, unit)) return;  // all threads of a spare CTA
    } else {
        bwd_cta_tile<MASK>(p, int(gridDim.y), kt, unit);
    }
    const KvUnit u = kv_unit(p, unit);
    const int b = u.b;
    int q_first = 0;
    const int n_per = bwd_q_count<MASK>(p, kt, q_first);  // query steps per query head
    const int n_it = n_per * u.nqh;                        // steps over all the unit's query heads

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(q_full + i, 2);
            mbar_init(q_empty + i, 1);
        }
        mbar_init(do_full, 1);
        mbar_init(do_empty, 1);
        mbar_init(s_full, 1);
        mbar_init(dp_full, 1);
        mbar_init(p_full, 8);
        mbar_init(ds_full, 8);
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

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        // Q (with the step's lse and Delta) is double-buffered; dO has one slot, refilled
        // as soon as dV of the previous step has read it, well before the next dP^T needs it
        bool ok = true;
        int nq = 0, ndo = 0;
        if (n_it > 0) {
            if (lane == 0) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
                tma_prefetch_desc(&tm_do);
                mbar_arrive_expect_tx(kv_full, 2 * C::T_BYTES);
                kv_load<D>(sK, &tm_k, kv_full, p, kt * kTile, u);
                kv_load<D>(sV, &tm_v, kv_full, p, kt * kTile, u);
            }
            // lse and Delta arrive by bulk copy when the step is whole and 16-byte aligned
            const bool bulk_stats = (p.L % 4) == 0;
            for (int it = 0; it < n_it; ++it) {
                const int qs = it & 1;
                if (it >= 2) {
                    ok = __all_sync(0xffffffffu, mbar_wait(q_empty + qs, ((it >> 1) - 1) & 1, ab, ROLE_LOAD, 1));
                    if (!ok) break;
                }
                const int ih = it / n_per;
                const int h = u.h_first + ih;
                const int q0 = bwd_q_step<MASK>(p, q_first, it - ih * n_per) * kQStep;
                const bool whole = bulk_stats && q0 + kQStep <= p.L;
                // Q by TMA; lse and Delta by the warp's lanes (two 16-byte loads each, both in
                // flight before either store), so that the TMA queue carries two instructions
                // per Q tile instead of four. The slot's barrier takes both arrivals.
                if (lane == 0) {
                    mbar_arrive_expect_tx(q_full + qs, C::T_BYTES);
                    bwd_load<D>(sQ + qs * C::T_BYTES, &tm_q, q_full + qs, p, q0, h, b);
                }
                if (whole) {
                    const float4 l4 = reinterpret_cast<const float4*>(p.lse + stat_index(p, q0, h, b))[lane];
                    const float4 d4 = reinterpret_cast<const float4*>(p.delta + stat_index(p, q0, h, b))[lane];
                    reinterpret_cast<float4*>(sLSE + qs * kQStep)[lane] = l4;
                    reinterpret_cast<float4*>(sDelta + qs * kQStep)[lane] = d4;
                } else {
                    for (int c = lane; c < kQStep; c += 32) {
                        const int q = q0 + c;
                        const bool in = q < p.L;
                        // rows past the end get lse = +inf, hence P = 0
                        sLSE[qs * kQStep + c] = in ? p.lse[stat_index(p, q, h, b)] : INFINITY;
                        sDelta[qs * kQStep + c] = in ? p.delta[stat_index(p, q, h, b)] : 0.f;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(q_full + qs);
                ++nq;
                if (it >= 1) {
                    ok = __all_sync(0xffffffffu, mbar_wait(do_empty, (it - 1) & 1, ab, ROLE_LOAD, 2));
                    if (!ok) break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(do_full, C::T_BYTES);
                    bwd_load<D>(sDO, &tm_do, do_full, p, q0, h, b);
                }
                ++ndo;
            }
            if (!ok && lane == 0) {
                mbar_drain(kv_full, 0);
                for (int qs = 0; qs < 2; ++qs) {
                    const int cnt = nq > qs ? (nq - 1 - qs) / 2 + 1 : 0;
                    if (cnt > 0) mbar_drain(q_full + qs, (cnt - 1) & 1);
                }
                if (ndo > 0) mbar_drain(do_full, (ndo - 1) & 1);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0 && n_it > 0) {
            constexpr uint32_t id_s = idesc_bf16(128, kQStep, 0, 0);   // S^T, dP^T
            constexpr uint32_t id_kv = idesc_bf16(128, D, 0, 1);       // dV, dK
            constexpr uint32_t id_dq = idesc_bf16(128, kQStep, 1, 1);  // dQ^T (M padded to 128 for d=64)
            const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aQ = smem_u32(sQ), aDO = smem_u32(sDO);
            const uint32_t aDSt = smem_u32(sDSt);
            const uint32_t tS = tmem + C::T_S, tDP = tmem + C::T_DP, tDV = tmem + C::T_DV, tDK = tmem + C::T_DK;
            // descriptors at the operands' base addresses; k-steps move them by constant offsets
            const uint64_t dK_k = sdesc_sw128(aK, 16, 1024), dV_k = sdesc_sw128(aV, 16, 1024);
            const uint64_t dDO_k = sdesc_sw128(aDO, 16, 1024), dDO_mn = sdesc_sw128(aDO, C::CHUNK, 1024);
            // K^T as an MN-major A operand: the second 64-row block of M is the second d chunk.
            // With d = 64 that block reads the V tile behind K; those lanes of dQ^T are ignored.
            const uint64_t dKt_mn = sdesc_sw128(aK, C::CHUNK, 1024);
            const uint64_t dDSt_mn = sdesc_sw128(aDSt, C::DST_BYTES / 2, 1024);
            const uint64_t dDSt_k = sdesc_sw128(aDSt, 16, 1024);
            auto issue_s = [&](int j) {  // S^T = K Q^T
                const uint64_t dQ_k = sdesc_sw128(aQ + (j & 1) * C::T_BYTES, 16, 1024);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t o = (k >> 2) * C::CHUNK + (k & 3) * 32;
                    umma_ss(tS, sdesc_add(dK_k, o), sdesc_add(dQ_k, o), id_s, k > 0);
                }
                umma_commit(s_full);
            };
            auto issue_dp = [&]() {  // dP^T = V dO^T
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t o = (k >> 2) * C::CHUNK + (k & 3) * 32;
                    umma_ss(tDP, sdesc_add(dV_k, o), sdesc_add(dDO_k, o), id_s, k > 0);
                }
                umma_commit(dp_full);
            };

            bool ok = mbar_wait(kv_full, 0, ab, ROLE_MMA, 1) && mbar_wait(q_full, 0, ab, ROLE_MMA, 2) &&
                      mbar_wait(do_full, 0, ab, ROLE_MMA, 3);
            if (ok) {
                tc_fence_after();
                issue_s(0);
                issue_dp();
            }
            // Per step: dV, then the next S^T (so that the softmax warps compute the next P
            // while dK and dQ^T run), dK, dQ^T over dS^T in the dP^T columns, and the next
            // dP^T once the softmax warps have read dQ^T out of those columns.
            for (int it = 0; ok && it < n_it; ++it) {
                const uint64_t dQ_mn = sdesc_sw128(aQ + (it & 1) * C::T_BYTES, C::CHUNK, 1024);
                const bool more = it + 1 < n_it;
                // dV += P^T dO  (P^T bf16 over S^T)
                if (!(ok = mbar_wait(p_full, it & 1, ab, ROLE_MMA, 4))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < kQStep / 16; ++k)
                    umma_ts(tDV, tS + a_col(k), sdesc_add(dDO_mn, k * 2048), id_kv, (it > 0 || k > 0) ? 1u : 0u);
                umma_commit(do_empty);
                // the next S^T over P^T: dV, which reads it, was issued first, and tcgen05
                // operations of one thread execute in order
                if (more) {
                    if (!(ok = mbar_wait(q_full + ((it + 1) & 1), ((it + 1) >> 1) & 1, ab, ROLE_MMA, 5))) break;
                    tc_fence_after();
                    issue_s(it + 1);
                }
                // dQ^T = K^T dS^T over the dP^T columns (the softmax warps have read dP^T), first,
                // so that the drain warps read it out while dK runs
                if (!(ok = mbar_wait(ds_full, it & 1, ab, ROLE_MMA, 6))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < kTile / 16; ++k)
                    umma_ss(tDP, sdesc_add(dKt_mn, k * 2048), sdesc_add(dDSt_mn, k * 2048), id_dq, k > 0 ? 1u : 0u);
                umma_commit(dq_full);
                // dK += dS^T Q: dS^T from shared memory as a K-major A operand (its rows are keys
                // with 64 queries per 128 bytes, the layout the dQ^T MMA reads as MN-major B)
#pragma unroll
                for (int k = 0; k < kQStep / 16; ++k) {
                    const uint32_t o = (k >> 2) * (C::DST_BYTES / 2) + (k & 3) * 32;
                    umma_ss(tDK, sdesc_add(dDSt_k, o), sdesc_add(dQ_mn, k * 2048), id_kv, (it > 0 || k > 0) ? 1u : 0u);
                }
                umma_commit(q_empty + (it & 1));
                if (more) {
                    // the next dP^T overwrites dQ^T: wait until the drain warps have read it
                    if (!(ok = mbar_wait(dq_free, it & 1, ab, ROLE_MMA, 7))) break;
                    if (!(ok = mbar_wait(do_full, (it + 1) & 1, ab, ROLE_MMA, 8))) break;
                    tc_fence_after();
                    issue_dp();
                }
            }
            if (ok) umma_commit(dkdv_done);
            else {
                umma_commit(drain);
                mbar_drain(drain, 0);
            }
        }
    } else if (warp < 10) {
        // ------------------------------------------------------------------ softmax, dS
        // thread = one key (tensor-memory lane); half hf takes queries [64 hf, 64 hf + 64)
        const int wq = warp & 3;
        const int hf = (warp - 2) >> 2;
        const int row = wq * 32 + lane;
        const uint32_t lane_off = uint32_t(wq * 32) << 16;
        const int key = kt * kTile + row;
        // this warp's chunk of the dS^T buffer (64 queries of every key)
        const uint32_t dst_chunk = smem_u32(sDSt) + hf * (C::DST_BYTES / 2);
        bool ok = true;
        // Per step: dS of this step, then P of the next step (whose S^T the MMA issuer
        // started right after this step's dV, so that its exponentials overlap dK and dQ^T).
        // P is kept in registers (fp32) from its computation until dS uses it.
        float pv[64];
        // P = exp(scale S - lse) of step j over S^T, written back as bf16 P^T (A operand of dV)
        auto softmax_p = [&](int j) -> bool {
            const int qs = j & 1;
            const int jh = j / n_per;
            const int q0 = bwd_q_step<MASK>(p, q_first, j - jh * n_per) * kQStep + 64 * hf;
            if (!__all_sync(0xffffffffu, mbar_wait(q_full + qs, (j >> 1) & 1, ab, ROLE_SOFTMAX, 1) &&
                                             mbar_wait(s_full, j & 1, ab, ROLE_SOFTMAX, 2)))
                return false;
            tc_fence_after();
            tmem_ld32(tmem + C::T_S + lane_off + 64 * hf, pv);
            tmem_ld32(tmem + C::T_S + lane_off + 64 * hf + 32, pv + 32);
            tmem_wait_ld();
            // every lane needs the same 64 lse values: 16-byte broadcast loads (a quarter of
            // the shared-memory wavefronts of scalar ones, which compete with the MMA operands)
            const float4* lse4 = reinterpret_cast<const float4*>(sLSE + qs * kQStep + 64 * hf);
            const bool diag = (MASK == ULYSSES_MASK_CAUSAL) && (q0 < key);
#pragma unroll
            for (int c4 = 0; c4 < 16; ++c4) {
                const float4 l = lse4[c4];
                const float nl[4] = {-l.x * kLog2e, -l.y * kLog2e, -l.z * kLog2e, -l.w * kLog2e};
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const int c = 4 * c4 + x;
                    float e = ex2(fmaf(pv[c], p.scale_log2, nl[x]));
                    if (diag && q0 + c < key) e = 0.f;
                    pv[c] = e;
                }
            }
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) pk[i] = pack_bf16(pv[2 * i], pv[2 * i + 1]);
            tmem_st32_u(tmem + C::T_S + lane_off + 96 * hf, pk);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
            return true;
        };
        if (n_it > 0) ok = softmax_p(0);
        for (int it = 0; ok && it < n_it; ++it) {
            const int qs = it & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(dp_full, it & 1, ab, ROLE_SOFTMAX, 3));
            if (!ok) break;
            tc_fence_after();
            // dS = P (dP - Delta), 32 columns at a time to bound the live registers
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float dp[32];
                tmem_ld32(tmem + C::T_DP + lane_off + 64 * hf + 32 * hh, dp);
                tmem_wait_ld();
                const float4* dl4 = reinterpret_cast<const float4*>(sDelta + qs * kQStep + 64 * hf + 32 * hh);
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    const float4 dl = dl4[c4];
                    const float dv4[4] = {dl.x, dl.y, dl.z, dl.w};
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const int c = 32 * hh + 4 * c4 + x;
                        pv[c] = pv[c] * (dp[4 * c4 + x] - dv4[x]);
                    }
                }
            }
            {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) pk[i] = pack_bf16(pv[2 * i], pv[2 * i + 1]);
                // B operand of dQ^T and A operand of dK
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    st_shared_v4(dst_chunk + sw128_offset(row, u), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2],
                                 pk[4 * u + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(ds_full);

            if (it + 1 < n_it && !(ok = softmax_p(it + 1))) break;
        }
        // ------------------------------------------------------------------ dK, dV epilogue
        if (ok && n_it > 0) ok = __all_sync(0xffffffffu, mbar_wait(dkdv_done, 0, ab, ROLE_EPI, 1));
        if (ok) {
            tc_fence_after();
            // half 0 writes dV, half 1 writes dK
            const uint32_t tcol = hf == 0 ? C::T_DV : C::T_DK;
            const float mul = hf == 0 ? 1.0f : p.scale;
            const size_t koff = kv_row_offset(p, key, u, D);
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(hf == 0 ? p.dv : p.dk) + koff;
            const bool valid = key < p.L;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float x[32];
                if (n_it > 0) {
                    tmem_ld32(tmem + tcol + lane_off + c * 32, x);
                    tmem_wait_ld();
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) x[i] = (n_it > 0) ? x[i] * mul : 0.f;
                if constexpr (ACC) {
                    if (!valid) continue;
                    float4* a4 = reinterpret_cast<float4*>((hf == 0 ? p.dv_acc : p.dk_acc) + koff + c * 32);
                    if (p.dkv_mode >= 2) {
#pragma unroll
                        for (int y = 0; y < 8; ++y) {
                            const float4 t = a4[y];
                            x[4 * y] += t.x; x[4 * y + 1] += t.y; x[4 * y + 2] += t.z; x[4 * y + 3] += t.w;
                        }
                    }
                    if (p.dkv_mode <= 2) {
#pragma unroll
                        for (int y = 0; y < 8; ++y) a4[y] = make_float4(x[4 * y], x[4 * y + 1], x[4 * y + 2], x[4 * y + 3]);
                        continue;
                    }
                }
                if (valid) {
                    uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                    for (int y = 0; y < 4; ++y)
                        d4[y] = make_uint4(pack_bf16(x[8 * y], x[8 * y + 1]), pack_bf16(x[8 * y + 2], x[8 * y + 3]),
                                           pack_bf16(x[8 * y + 4], x[8 * y + 5]), pack_bf16(x[8 * y + 6], x[8 * y + 7]));
                }
            }
        }
    } else {
        // ------------------------------------------------------------------ dQ drain (warps 10-13)
        // Warp 10 + i reads dQ^T lanes [32 wq, 32 wq + 32) (features, wq = warp % 4, the lane
        // quadrant this warp may access) for all 128 queries of the step, 64 columns at a time,
        // and frees the columns for the next dP^T once both halves are in registers or staged.
        // Each half goes to the warp's 8 KB shared-memory slot in the accumulator's block layout
        // and is added into global memory by one bulk reduction on the TMA engine, so no warp
        // issues per-element reductions: those would queue in the same per-sub-partition memory
        // pipe as the softmax warps' shared-memory traffic and stretch their loop.
        const int wq = warp & 3;
        const uint32_t lane_off = uint32_t(wq * 32) << 16;
        const bool dq_lanes = wq * 32 < D;  // warp-uniform: d = 64 leaves quadrants 2, 3 without dQ rows
        const uint32_t slot = smem_u32(smem + C::OFF_STG + (warp - 10) * 8192);
        const uint32_t mine = slot + lane * 256;
        const uint32_t sw = uint32_t(lane & 7);
        bool ok = true;
        // one half: wait until the slot's previous bulk reduction has read it, stage, add
        auto stage_add = [&](const float* v, float* dst) {
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
#pragma unroll
            for (int u4 = 0; u4 < 16; ++u4)
                st_shared_v4(mine + ((uint32_t(u4) ^ sw) << 4), __float_as_uint(v[4 * u4]), __float_as_uint(v[4 * u4 + 1]),
                             __float_as_uint(v[4 * u4 + 2]), __float_as_uint(v[4 * u4 + 3]));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                bulk_reduce_add_f32(dst, slot, 8192);
                bulk_commit_group();
            }
        };
        for (int it = 0; ok && it < n_it; ++it) {
            const int ih = it / n_per;
            const int h = u.h_first + ih;
            const int qstep = bwd_q_step<MASK>(p, q_first, it - ih * n_per);
            ok = __all_sync(0xffffffffu, mbar_wait(dq_full, it & 1, ab, ROLE_DQ, 1));
            if (!ok) break;
            tc_fence_after();
            float v[64];
            tmem_ld32(tmem + C::T_DP + lane_off, v);
            tmem_ld32(tmem + C::T_DP + lane_off + 32, v + 32);
            tmem_wait_ld();
            float* acc = p.dq_acc + dq_block<D>(p, b * p.H + h, qstep, 0, wq) * kDqBlockFloats;
            if (dq_lanes) stage_add(v, acc);
            tmem_ld32(tmem + C::T_DP + lane_off + 64, v);
            tmem_ld32(tmem + C::T_DP + lane_off + 96, v + 32);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dq_free);
            if (dq_lanes) stage_add(v, acc + size_t(D / 32) * kDqBlockFloats);
        }
        // the reductions complete before the CTA (and its shared memory) goes away
        if (lane == 0) bulk_wait_all();
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
    // zero the fp32 dQ accumulator (padded to whole 128-row steps)
    const size_t n4 = size_t(p.B) * p.H * p.n_tiles * kTile * D / 4;
    float4* acc = reinterpret_cast<float4*>(p.dq_acc);
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += size_t(gridDim.x) * blockDim.x)
        acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// dQ = bf16(scale * accumulator), written in the output layout. One warp per (batch x head,
// query step, query half): the D/32 accumulator blocks of those 64 queries. Thread t takes
// features [8 o, 8 o + 8) with o = t % (D / 8) and every other 4-query unit; per unit it loads
// its 8 features' 16-byte units, transposes them in registers and writes four 16-byte rows
// pieces, so that the threads of one unit write whole contiguous rows.
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(BwdParams p, __nv_bfloat16* dq) {
    constexpr int NQ = D / 32;          // feature quadrants (blocks per group)
    constexpr int OCT = D / 8;          // feature octets: 16 for d = 128, 8 for d = 64
    constexpr int UPASS = 32 / OCT;     // 4-query units a warp covers at once: 2 or 4
    const size_t groups = size_t(p.B) * p.H * p.n_tiles * 2;
    const uint32_t lane = threadIdx.x & 31u;
    const int o = int(lane) % OCT;
    const int wq = o / 4;               // quadrant of this thread's features
    const int l0 = (o % 4) * 8;         // first feature lane within the quadrant block
    for (size_t grp = (size_t(blockIdx.x) * blockDim.x + threadIdx.x) / 32; grp < groups;
         grp += size_t(gridDim.x) * blockDim.x / 32) {
        const int hq = int(grp % 2);
        const size_t sb = grp / 2;  // (batch x head, query step)
        const int qstep = int(sb % p.n_tiles);
        const int bh = int(sb / p.n_tiles);
        const int h = bh % p.H, b = bh / p.H;
        const float* blk = p.dq_acc + (grp * NQ + wq) * kDqBlockFloats;
        const int s0 = qstep * kQStep + hq * 64;
        for (int u = int(lane) / OCT; u < 16; u += UPASS) {
            float x[8][4];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int l = l0 + i;
                const float4 v = reinterpret_cast<const float4*>(blk + l * 64)[uint32_t(u) ^ uint32_t(l & 7)];
                x[i][0] = v.x; x[i][1] = v.y; x[i][2] = v.z; x[i][3] = v.w;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int s = s0 + 4 * u + c;
                if (s >= p.L) continue;
                uint4 w;
                w.x = pack_bf16(x[0][c] * p.scale, x[1][c] * p.scale);
                w.y = pack_bf16(x[2][c] * p.scale, x[3][c] * p.scale);
                w.z = pack_bf16(x[4][c] * p.scale, x[5][c] * p.scale);
                w.w = pack_bf16(x[6][c] * p.scale, x[7][c] * p.scale);
                *reinterpret_cast<uint4*>(dq + row_offset(p, s, h, b, D) + 8 * o) = w;
            }
        }
    }
}

static size_t acc_bytes(const ulysses_shape_t& s) {
    const size_t rows = (size_t(s.L) + kTile - 1) / kTile * kTile;
    return (size_t(s.B) * s.H * rows * s.d_h * 4 + 255) / 256 * 256;
}

size_t bwd_workspace_bytes(const ulysses_shape_t& s) {
    const size_t rows = size_t(s.B) * s.H * s.L;
    const size_t n_tiles = (size_t(s.L) + kTile - 1) / kTile;
    return acc_bytes(s) + (rows * 4 + 255) / 256 * 256 + (4 * n_tiles * 4 + 255) / 256 * 256;
}

// Block-sparse schedule, step 1: each key tile's rank by (CSC length descending, index).
__global__ void __launch_bounds__(256) bwd_order_kernel(const int32_t* colptr, int n, int32_t* sched) {
    for (int kt = blockIdx.x * blockDim.x + threadIdx.x; kt < n; kt += gridDim.x * blockDim.x) {
        const int len = colptr[kt + 1] - colptr[kt];
        int rank = 0;
        for (int j = 0; j < n; ++j) {
            const int lj = colptr[j + 1] - colptr[j];
            rank += (lj > len || (lj == len && j < kt)) ? 1 : 0;
        }
        sched[rank] = kt;
        sched[n + rank] = len;
    }
}

// Step 2: for each position of the order, the start and size of its run of equal lengths
// (binary searches over the non-increasing lengths).
__global__ void __launch_bounds__(256) bwd_class_kernel(int n, int32_t* sched) {
    const int32_t* len = sched + n;
    for (int pos = blockIdx.x * blockDim.x + threadIdx.x; pos < n; pos += gridDim.x * blockDim.x) {
        const int l = len[pos];
        int lo = 0, hi = pos;  // first index with len == l
        while (lo < hi) {
            const int mid = (lo + hi) / 2;
            if (len[mid] > l) lo = mid + 1; else hi = mid;
        }
        int lo2 = pos, hi2 = n;  // first index with len < l
        while (lo2 < hi2) {
            const int mid = (lo2 + hi2) / 2;
            if (len[mid] >= l) lo2 = mid + 1; else hi2 = mid;
        }
        sched[2 * n + pos] = lo;
        sched[3 * n + pos] = lo2 - lo;
    }
}

template <int D, int MASK, bool ACC>
static int launch_bwd_t(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mdo,
                        const BwdParamsOf<ACC>& p, cudaStream_t stream) {
    using C = BwdCfg<D>;
    // one CTA per (key tile, key/value head unit): B * Hkv units token-sharded, P * B * Hkvp head-sharded
    const int units = p.layout == ULYSSES_LAYOUT_TOKEN_SHARDED ? p.B * p.Hkv : p.P * p.B * p.Hkvp;
    int G = 1;
    if (MASK == ULYSSES_MASK_CAUSAL) {
        // per unit: its query heads' Q and dO (bf16) and dQ accumulator (fp32)
        const int nqh = p.layout == ULYSSES_LAYOUT_TOKEN_SHARDED ? p.G : (p.kv_rep == 1 ? p.G : p.Hp);
        const size_t unit_bytes = size_t(p.L) * D * 8 * size_t(nqh);
        G = int(std::min<size_t>(size_t(units), std::max<size_t>(1, (size_t(32) << 20) / unit_bytes)));
    }
    // the grouped order is a kernel of its own: the plain kernel's code stays as it is (the
    // backward measurably slowed when its mapping code grew)
    auto kern = G > 1 ? attn_bwd_kernel<D, MASK, ACC, true> : attn_bwd_kernel<D, MASK, ACC, false>;
    if (!set_max_dynamic_smem(reinterpret_cast<const void*>(kern), C::SMEM_BYTES)) return ULYSSES_ERR_CUDA;
    dim3 grid(G * p.n_tiles, (units + G - 1) / G);
    kern<<<grid, kBwdThreads, C::SMEM_BYTES, stream>>>(mq, mk, mv, mdo, p);
    return cudaGetLastError() == cudaSuccess ? ULYSSES_OK : ULYSSES_ERR_CUDA;
}

template <int D>
static int launch_bwd_d(const ulysses_shape_t& s, const MaskArgs& m, BwdParams& p, const void* q, const void* k,
                        const void* v, const void* o, const void* dO, void* dq, const BwdChain& chain,
                        cudaStream_t stream) {
    CUtensorMap mq, mk, mv, mdo;
    if (!encode_qkv_map(&mq, q, s, p.layout, p.box_rows, s.H, s.H / s.P) ||
        !encode_qkv_map(&mdo, dO, s, p.layout, p.box_rows, s.H, s.H / s.P) ||
        !encode_qkv_map(&mk, k, s, p.layout, p.box_rows, p.Hkv, p.Hkvp) ||
        !encode_qkv_map(&mv, v, s, p.layout, p.box_rows, p.Hkv, p.Hkvp))
        return ULYSSES_ERR_CUDA;
    const int sms = device_sm_count();
    const size_t rows = size_t(s.B) * s.H * s.L;
    size_t blocks = (rows * 8 + 255) / 256;
    if (blocks > size_t(sms) * 16) blocks = size_t(sms) * 16;
    if (chain.prep) {
        bwd_prep_kernel<D><<<unsigned(blocks), 256, 0, stream>>>(p, static_cast<const __nv_bfloat16*>(o),
                                                                  static_cast<const __nv_bfloat16*>(dO),
                                                                  const_cast<float*>(p.delta));
        if (cudaGetLastError() != cudaSuccess) return ULYSSES_ERR_CUDA;
    }
    if (m.kind == ULYSSES_MASK_BLOCK_SPARSE) {
        int32_t* sched = reinterpret_cast<int32_t*>(const_cast<float*>(p.delta) + (rows + 63) / 64 * 64);
        const unsigned ob = unsigned((p.n_tiles + 255) / 256);
        bwd_order_kernel<<<ob, 256, 0, stream>>>(p.colptr, p.n_tiles, sched);
        bwd_class_kernel<<<ob, 256, 0, stream>>>(p.n_tiles, sched);
        if (cudaGetLastError() != cudaSuccess) return ULYSSES_ERR_CUDA;
    }
    int rc;
    if (chain.dkv_mode != 0) {
        BwdAccParams ap;
        static_cast<BwdParams&>(ap) = p;
        ap.dk_acc = chain.dk_acc;
        ap.dv_acc = chain.dv_acc;
        ap.dkv_mode = chain.dkv_mode;
        // the accumulating epilogue is built for the masks of the ring blocks only
        if (m.kind == ULYSSES_MASK_CAUSAL) rc = launch_bwd_t<D, ULYSSES_MASK_CAUSAL, true>(mq, mk, mv, mdo, ap, stream);
        else if (m.kind == ULYSSES_MASK_NONE) rc = launch_bwd_t<D, ULYSSES_MASK_NONE, true>(mq, mk, mv, mdo, ap, stream);
        else return ULYSSES_ERR_UNSUPPORTED;
    } else if (m.kind == ULYSSES_MASK_CAUSAL) rc = launch_bwd_t<D, ULYSSES_MASK_CAUSAL, false>(mq, mk, mv, mdo, p, stream);
    else if (m.kind == ULYSSES_MASK_NONE) rc = launch_bwd_t<D, ULYSSES_MASK_NONE, false>(mq, mk, mv, mdo, p, stream);
    else rc = launch_bwd_t<D, ULYSSES_MASK_BLOCK_SPARSE, false>(mq, mk, mv, mdo, p, stream);
    if (rc != ULYSSES_OK) return rc;
    if (!chain.convert) return ULYSSES_OK;
    bwd_dq_convert_kernel<D><<<unsigned(blocks), 256, 0, stream>>>(p, static_cast<__nv_bfloat16*>(dq));
    return cudaGetLastError() == cudaSuccess ? ULYSSES_OK : ULYSSES_ERR_CUDA;
}

int launch_attn_bwd(const ulysses_shape_t& s, const MaskArgs& m, float scale, int layout, const void* q,
                    const void* k, const void* v, const void* o, const float* lse, const void* dO, void* dq,
                    void* dk, void* dv, void* workspace, cudaStream_t stream, const BwdChain& chain) {
    BwdParams p{};
    p.B = s.B; p.L = s.L; p.H = s.H; p.P = s.P; p.Hp = s.H / s.P; p.Lp = s.L / s.P;
    const KvInfo kv = kv_info(s);
    p.Hkv = kv.Hkv; p.G = kv.G; p.Hkvp = kv.Hkvp; p.kv_rep = kv.rep;
    p.layout = layout;
    p.n_tiles = (s.L + kTile - 1) / kTile;
    p.box_rows = layout == ULYSSES_LAYOUT_TOKEN_SHARDED ? gcd_int(p.Lp, kTile) : kTile;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.lse = lse;
    p.dq_acc = static_cast<float*>(workspace);
    p.delta = reinterpret_cast<float*>(static_cast<char*>(workspace) + acc_bytes(s));
    p.dk = dk;
    p.dv = dv;
    if (chain.dkv_mode < 0 || chain.dkv_mode > 3 || (chain.dkv_mode != 0 && (!chain.dk_acc || !chain.dv_acc)))
        return ULYSSES_ERR_INVALID_ARG;
    p.colptr = m.k_colptr;
    p.qrows = m.k_qrows;
    p.err = device_error_word();
    if (!p.err) return ULYSSES_ERR_CUDA;
    if (s.d_h == 128) return launch_bwd_d<128>(s, m, p, q, k, v, o, dO, dq, chain, stream);
    return launch_bwd_d<64>(s, m, p, q, k, v, o, dO, dq, chain, stream);
}

}  // namespace ulysses
