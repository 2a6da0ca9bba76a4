// The projections on either side of the Ulysses attention block (paper summary section 3.2
// "Big-Picture Architecture" and section 3.4.1 "Before attention"; pinyu.ai page "One
// attention block, end to end"): each rank projects its own token shard to Q, K, V before
// the first all-to-all, and projects the returned O after the second. Every token row is
// projected on its own, so on the token-sharded layout [P][B][Lp][features] both are one
// matrix product over the rows, C[M][N] = A[M][K] B[N][K]^T (M = B L token rows, weights
// in the y = x W^T convention):
//   QKV projection:  A = X [M][hidden], B = W_qkv [(H + 2 Hkv) d][hidden]; the epilogue
//                    writes columns [0, H d) to Q, [H d, (H + Hkv) d) to K and the rest
//                    to V, each row-major, i.e. directly in the token-sharded layout the
//                    attention kernels read (no relayout pass);
//   out projection:  A = O [M][H d], B = W_o [hidden][H d], C = Y [M][hidden].
//
// Persistent CTA pairs (clusters of two on neighbouring SMs) walk 256 x 256 tiles of C on the
// 5th-generation tensor cores with paired-SM MMAs (tcgen05 cta_group::2): each CTA holds 128
// rows of A and its 128-row half of B, and the pair's M256 N256 K16 MMA, issued by the
// leader, reads both CTAs' shared memory and writes each CTA's 128 rows into its own tensor
// memory. Per SM that halves the B operand's loads and shared-memory reads against a 1-SM
// 128 x 256 tile, whose traffic (about 190 B/clk) exceeded the 128 B/clk shared-memory port.
//   warp 0 (both CTAs) loads A and B K-slices of 128 through a 3-stage TMA ring that runs on
//          across tiles, one copy per operand and slice (both 64-wide chunks: the per-SM TMA
//          engine moves larger copies faster); both CTAs' loads count on the leader's barrier;
//   warp 1 (leader) issues the MMAs into one of two TMEM accumulators (256 columns each) and
//          commits to the barriers of both CTAs at once;
//   warps 2-5 (both CTAs) convert the other accumulator to bf16 and store their rows, so a
//          tile's epilogue overlaps the next tile's MMAs.
// Tiles are rasterized in groups of 8 row tiles (16 when B exceeds 48 MB), so the tiles in
// flight at one time share their A and B slices in L2.
#include <mutex>

#include "common.cuh"
#include "ulysses_internal.h"

namespace ulysses {

struct GemmCfg {
    // a CTA pair computes a 256 x 256 tile; each CTA holds 128 rows of A and 128 rows of B
    // K-slices of 128: one TMA copy brings both 64-wide chunks of a 128-row slice (32 KB)
    static constexpr int BM = 128, BN = 256, BK = 128, STAGES = 3;
    static constexpr int PM = 2 * BM;                  // pair tile rows
    static constexpr uint32_t CHUNK = 128 * 128;       // 128 rows x 64 elements, swizzled
    static constexpr uint32_t A_BYTES = BM * BK * 2;   // 32 KB
    static constexpr uint32_t B_BYTES = (BN / 2) * BK * 2;  // 32 KB: this CTA's half of B
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t OFF_BAR = STAGES * STAGE_BYTES;
    static constexpr uint32_t SMEM_BYTES = OFF_BAR + 256 + 1024;
    static constexpr uint32_t TMEM_COLS = 512;  // two accumulators of 256 columns
    static constexpr int kThreads = 192;
};

struct GemmParams {
    int M, N, K;
    int n_out;          // column ranges of C written to separate outputs (1 or 3)
    int col0[4];        // range i is columns [col0[i], col0[i + 1])
    void* out[3];       // bf16, row-major
    int ld[3];          // row pitch of each output in elements
    int chunked;        // 1: the maps bring a whole 128-wide K slice per copy (K % 64 == 0)
    int group_m;        // row tiles per raster group
    uint32_t* err;
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GemmCfg::kThreads, 1)
proj_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, const GemmParams p) {
    using C = GemmCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* full = bars;                  // [STAGES], the leader's counts both CTAs' loads
    uint64_t* empty = bars + C::STAGES;     // [STAGES], both CTAs (multicast commit)
    uint64_t* acc_full = bars + 2 * C::STAGES;   // [2], both CTAs (multicast commit)
    uint64_t* acc_empty = acc_full + 2;          // [2], the leader's: 4 epilogue warps of each CTA
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = static_cast<int>(warp_id());
    const int lane = static_cast<int>(lane_id());
    const uint32_t rank = cluster_rank();    // 0: the leader, which issues the pair's MMAs
    const int pair = blockIdx.x / 2, n_pairs = gridDim.x / 2;
    const int tiles_m = (p.M + C::PM - 1) / C::PM, tiles_n = (p.N + C::BN - 1) / C::BN;
    const int n_tiles = tiles_m * tiles_n;
    const int n_k = (p.K + C::BK - 1) / C::BK;
    // grouped raster: group_m row tiles vary fastest, then column tiles, then groups
    auto tile_origin = [&](int t, int& m0, int& n0) {
        const int per_group = p.group_m * tiles_n;
        const int group = t / per_group;
        const int gm = min(p.group_m, tiles_m - group * p.group_m);  // row tiles in this group
        const int in_group = t - group * per_group;
        m0 = (group * p.group_m + in_group % gm) * C::PM;
        n0 = (in_group / gm) * C::BN;
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(acc_full + i, 1);
            mbar_init(acc_empty + i, 8);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    tc_fence_before();
    // both CTAs' barriers exist before either CTA signals the other's
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Abort ab{abort_flag, p.err, KID_PROJ};

    if (warp == 0) {
        // ------------------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            tma_prefetch_desc(&tm_a);
            tma_prefetch_desc(&tm_b);
            int issued = 0;  // K-slices loaded so far, over all of this pair's tiles
            bool ok = true;
            for (int t = pair; ok && t < n_tiles; t += n_pairs) {
                int m0, n0;
                tile_origin(t, m0, n0);
                for (int ks = 0; ks < n_k; ++ks, ++issued) {
                    const int s = issued % C::STAGES;
                    if (issued >= C::STAGES &&
                        !(ok = mbar_wait_cl(empty + s, ((issued / C::STAGES) - 1) & 1, ab, ROLE_LOAD, 1)))
                        break;
                    uint8_t* st = smem + s * C::STAGE_BYTES;
                    // both CTAs' bytes count on the leader's barrier; the leader expects them all
                    if (rank == 0) mbar_arrive_expect_tx(full + s, 2 * C::STAGE_BYTES);
                    const uint32_t lbar = cluster_addr(full + s, 0);
                    const int ra = m0 + int(rank) * C::BM, rb = n0 + int(rank) * (C::BN / 2);
                    if (p.chunked) {
                        tma_load_5d_pair(st, &tm_a, lbar, 0, ra, ks * (C::BK / 64), 0, 0);
                        tma_load_5d_pair(st + C::A_BYTES, &tm_b, lbar, 0, rb, ks * (C::BK / 64), 0, 0);
                    } else {
                        // a ragged K: 2-D boxes, whose columns past K read zeros
                        for (int c = 0; c < C::BK / 64; ++c) {
                            tma_load_2d_pair(st + c * C::CHUNK, &tm_a, lbar, ks * C::BK + c * 64, ra);
                            tma_load_2d_pair(st + C::A_BYTES + c * C::CHUNK, &tm_b, lbar, ks * C::BK + c * 64, rb);
                        }
                    }
                }
            }
            if (!ok) {
                // wait (bounded) for this CTA's stages' last loads to land: the leader's barrier
                // tracks them, so only the leader can; the peer waits on its empty barriers
                if (rank == 0) {
                    for (int s = 0; s < C::STAGES; ++s) {
                        const int cnt = issued > s ? (issued - 1 - s) / C::STAGES + 1 : 0;
                        if (cnt > 0) mbar_drain(full + s, (cnt - 1) & 1);
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer (leader)
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = idesc_bf16(C::PM, C::BN, 0, 0);
            const uint32_t base = smem_u32(smem);
            bool ok = true;
            int used = 0;  // K-slices consumed so far
            for (int t = pair, i = 0; ok && t < n_tiles; t += n_pairs, ++i) {
                const int a = i & 1;
                // both CTAs' epilogues must have read this accumulator's previous tile
                if (i >= 2 && !(ok = mbar_wait_cl(acc_empty + a, ((i >> 1) - 1) & 1, ab, ROLE_MMA, 2))) break;
                tc_fence_after();
                const uint32_t acc = tmem + a * C::BN;
                for (int ks = 0; ks < n_k; ++ks, ++used) {
                    const int s = used % C::STAGES;
                    if (!(ok = mbar_wait_cl(full + s, (used / C::STAGES) & 1, ab, ROLE_MMA, 1))) break;
                    tc_fence_after();
                    const uint64_t da = sdesc_sw128(base + s * C::STAGE_BYTES, 16, 1024);
                    const uint64_t db = sdesc_sw128(base + s * C::STAGE_BYTES + C::A_BYTES, 16, 1024);
#pragma unroll
                    for (int k = 0; k < C::BK / 16; ++k) {
                        const uint32_t o = (k >> 2) * C::CHUNK + (k & 3) * 32;
                        umma_pair_ss(acc, sdesc_add(da, o), sdesc_add(db, o), idesc, (ks > 0 || k > 0) ? 1u : 0u);
                    }
                    umma_pair_commit_both(empty + s);
                }
                if (ok) umma_pair_commit_both(acc_full + a);
            }
            if (!ok) {
                umma_pair_commit_both(drain);
                mbar_drain(drain, 0);
            }
        }
    } else {
        // ------------------------------------------------------------------ epilogue (both CTAs)
        // thread = one row of this CTA's 128 rows of the pair tile (TMEM lane); 32-column
        // chunks go to the output that holds them (the column ranges are multiples of 32 wide)
        const int wq = warp & 3;
        const uint32_t lane_off = uint32_t(wq * 32) << 16;
        const uint32_t lacc_empty0 = cluster_addr(acc_empty, 0);
        for (int t = pair, i = 0; n_k > 0 && t < n_tiles; t += n_pairs, ++i) {
            const int a = i & 1;
            int m0, n0;
            tile_origin(t, m0, n0);
            if (!__all_sync(0xffffffffu, mbar_wait_cl(acc_full + a, (i >> 1) & 1, ab, ROLE_EPI, 1))) break;
            tc_fence_after();
            const int row = m0 + int(rank) * C::BM + wq * 32 + lane;
            const uint32_t acc = tmem + lane_off + a * C::BN;
#pragma unroll 1
            for (int c = 0; c < C::BN; c += 32) {
                const int col = n0 + c;
                if (col >= p.N) break;  // warp-uniform
                float v[32];
                tmem_ld32(acc + c, v);
                tmem_wait_ld();
                int o = 0;
                while (o + 1 < p.n_out && col >= p.col0[o + 1]) ++o;
                if (row < p.M) {
                    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out[o]) + size_t(row) * p.ld[o] + (col - p.col0[o]);
                    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
                    for (int x = 0; x < 4; ++x)
                        d4[x] = make_uint4(pack_bf16(v[8 * x], v[8 * x + 1]), pack_bf16(v[8 * x + 2], v[8 * x + 3]),
                                           pack_bf16(v[8 * x + 4], v[8 * x + 5]), pack_bf16(v[8 * x + 6], v[8 * x + 7]));
                }
            }
            // this accumulator may take the next tile but one (the leader counts both CTAs)
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(lacc_empty0 + uint32_t(a) * 8u);
        }
    }

    tc_fence_before();
    __syncwarp();
    // the pair's MMAs and both CTAs' TMEM reads are over before either CTA frees the columns
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, C::TMEM_COLS);
    }
}

// 2-D bf16 tensor map over a row-major [rows][cols] matrix with a (64, box_rows) box and the
// 128-byte swizzle, zero fill out of bounds.
// Tensor map over a row-major [rows][cols] bf16 matrix, 128-byte swizzle, zero fill out of bounds.
// chunked (cols % 64 == 0): 5-D (64 elements, rows, 64-wide column chunks, 1, 1) with a box of
// box_rows rows of two chunks, chunk after chunk, so that one copy brings a 128-wide K slice (a
// chunk past the last column reads zeros). Otherwise 2-D (cols, rows) with a (64, box_rows) box.
static bool encode_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows, bool chunked) {
    if (chunked) {
        cuuint64_t dims[5] = {64, rows, cols / 64, 1, 1};
        cuuint64_t strides[4] = {cols * 2, 128, cols * 2 * rows, cols * 2 * rows};
        cuuint32_t box[5] = {64, box_rows, 2, 1, 1};
        cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        return encode_tensor_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, strides, box, estr);
    }
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return encode_tensor_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr);
}

int launch_proj_gemm(int M, int N, int K, const void* a, const void* b, int n_out, const int* col0, void* const* out,
                     const int* ld, cudaStream_t stream) {
    using C = GemmCfg;
    GemmParams p{};
    p.M = M; p.N = N; p.K = K; p.n_out = n_out;
    for (int i = 0; i <= n_out; ++i) p.col0[i] = col0[i];
    for (int i = 0; i < n_out; ++i) { p.out[i] = out[i]; p.ld[i] = ld[i]; }
    p.err = device_error_word();
    if (!p.err) return ULYSSES_ERR_CUDA;
    CUtensorMap ma, mb;
    // each CTA of a pair loads 128 rows of A and 128 rows (its half) of B per K-slice
    p.chunked = K % 64 == 0 ? 1 : 0;
    // every raster group reads all of B: when B is large, taller groups read it fewer times
    p.group_m = size_t(N) * size_t(K) * 2 > (size_t(48) << 20) ? 16 : 8;
    if (!encode_2d(&ma, a, uint64_t(M), uint64_t(K), C::BM, p.chunked) ||
        !encode_2d(&mb, b, uint64_t(N), uint64_t(K), C::BN / 2, p.chunked))
        return ULYSSES_ERR_CUDA;
    if (!set_max_dynamic_smem(reinterpret_cast<const void*>(proj_gemm_kernel), C::SMEM_BYTES)) return ULYSSES_ERR_CUDA;
    const int tiles = ((M + C::PM - 1) / C::PM) * ((N + C::BN - 1) / C::BN);
    // persistent: as many CTA pairs as can be resident at once (a pair needs two SMs of one
    // cluster-capable group; asked of the runtime once per device)
    static std::mutex mu;
    static int resident[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ULYSSES_ERR_CUDA;
    int pairs;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (resident[dev] == 0) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(unsigned(device_sm_count() / 2 * 2));
            cfg.blockDim = dim3(C::kThreads);
            cfg.dynamicSmemBytes = C::SMEM_BYTES;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, proj_gemm_kernel, &cfg) != cudaSuccess || n <= 0) return ULYSSES_ERR_CUDA;
            resident[dev] = n;
        }
        pairs = resident[dev];
    }
    if (tiles < pairs) pairs = tiles;
    proj_gemm_kernel<<<2 * pairs, C::kThreads, C::SMEM_BYTES, stream>>>(ma, mb, p);
    return cudaGetLastError() == cudaSuccess ? ULYSSES_OK : ULYSSES_ERR_CUDA;
}

}  // namespace ulysses
