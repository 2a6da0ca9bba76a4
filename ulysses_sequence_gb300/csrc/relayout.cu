// Standalone sequence<->head relayouts (the two all-to-alls of DeepSpeed-Ulysses, paper
// summary section 3.4.1; pinyu.ai page "Use the other independent axis"), as on-device
// permutations between the token-sharded [P][B][Lp][H][d] and head-sharded
// [P][B][L][Hp][d] layouts.
//
// Both layouts keep one head group of one token contiguous: a "run" of Hp*d elements.
// seq->head moves run (r, b, t, g) from in[((r*B + b)*Lp + t)*H*d + g*Hp*d] to
// out[((g*B + b)*L + r*Lp + t)*Hp*d]; head->seq moves it back. Runs are at least 256 bytes
// at every workload size, so 16-byte vector loads and stores are coalesced on both sides
// without staging: a warp copies whole token rows, with index arithmetic once per row.
#include <type_traits>

#include "common.cuh"
#include "ulysses_internal.h"

namespace ulysses {

struct RelayoutArgs {
    const void* in;
    void* out;
    uint32_t P, B, Lp, L, H, d;
    uint32_t G;          // head groups (P for the relayouts; any divisor of H for one rank's packing)
    uint32_t rows;       // token rows P * B * Lp
    uint32_t row_vecs;   // H * d / 8: 16-byte vectors of one token row (P runs)
    uint32_t run_vecs;   // Hp * d / 8: 16-byte vectors of one run
    int to_head;         // 1: seq->head, 0: head->seq
};

// A warp copies whole token rows (r, b, t): the token side of a row is contiguous, and
// vector w of the row belongs to group g = w / run_vecs, which lands at
// head[((g*B + b)*L + s)*run_vecs + w % run_vecs]. Each lane keeps the group offsets of
// its VPL vectors in registers, so a row costs two integer divisions in total.
template <int VPL, int UNROLL>
__global__ void __launch_bounds__(256, 2) relayout_row_kernel(RelayoutArgs a) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
    const uint32_t gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint4* __restrict__ in = static_cast<const uint4*>(a.in);
    uint4* __restrict__ out = static_cast<uint4*>(a.out);
    // a tensor holds fewer than 2^32 vectors (checked by the launcher), so 32 bits suffice
    const uint32_t group_stride = a.B * a.L * a.run_vecs;

    uint32_t goff[VPL];
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
        const uint32_t w = lane + 32u * k;
        const uint32_t g = w / a.run_vecs;
        goff[k] = g * group_stride + (w - g * a.run_vecs);
    }
    const uint32_t BLp = a.B * a.Lp;

    for (uint32_t row0 = gw * UNROLL; row0 < a.rows; row0 += nwarps * UNROLL) {
        uint4 v[UNROLL][VPL];
        uint64_t tok[UNROLL], head[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const uint32_t row = row0 + u;
            const uint32_t rr = row < a.rows ? row : 0;
            const uint32_t r = rr / BLp;
            const uint32_t rem = rr - r * BLp;
            const uint32_t b = rem / a.Lp;
            const uint32_t t = rem - b * a.Lp;
            tok[u] = uint64_t(rr) * a.row_vecs;
            head[u] = (uint64_t(b) * a.L + uint64_t(r) * a.Lp + t) * a.run_vecs;
            if (row < a.rows) {
#pragma unroll
                for (int k = 0; k < VPL; ++k) {
                    const uint32_t w = lane + 32u * k;
                    if (w < a.row_vecs) {
                        const uint64_t src = a.to_head ? tok[u] + w : head[u] + goff[k];
                        v[u][k] = __ldcs(in + src);
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            if (row0 + u < a.rows) {
#pragma unroll
                for (int k = 0; k < VPL; ++k) {
                    const uint32_t w = lane + 32u * k;
                    if (w < a.row_vecs) {
                        const uint64_t dst = a.to_head ? head[u] + goff[k] : tok[u] + w;
                        __stcs(out + dst, v[u][k]);
                    }
                }
            }
        }
    }
}

// Fallback for shapes whose runs are not whole 16-byte vectors or buffers not 16-byte
// aligned: one 2-byte element per thread.
__global__ void relayout_elem_kernel(RelayoutArgs a, uint64_t total) {
    const uint16_t* in = static_cast<const uint16_t*>(a.in);
    uint16_t* out = static_cast<uint16_t*>(a.out);
    const uint64_t run_elems = uint64_t(a.H / a.G) * a.d;
    for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += uint64_t(gridDim.x) * blockDim.x) {
        const uint64_t run = i / run_elems;
        const uint64_t e = i - run * run_elems;
        const uint64_t row = run / a.G;
        const uint64_t g = run - row * a.G;
        const uint64_t rb = row / a.Lp;
        const uint64_t t = row - rb * a.Lp;
        const uint64_t r = rb / a.B;
        const uint64_t b = rb - r * a.B;
        const uint64_t tok = i;
        const uint64_t head = ((g * a.B + b) * a.L + r * a.Lp + t) * run_elems + e;
        if (a.to_head) out[head] = in[tok];
        else out[tok] = in[head];
    }
}

int launch_relayout(const ulysses_shape_t& s, const void* in, void* out, cudaStream_t stream, bool to_head, int G) {
    RelayoutArgs a{};
    a.in = in;
    a.out = out;
    if (G <= 0) G = s.P;
    a.P = s.P; a.B = s.B; a.L = s.L; a.Lp = s.L / s.P; a.H = s.H; a.d = s.d_h; a.G = uint32_t(G);
    a.to_head = to_head ? 1 : 0;
    const uint64_t rows = uint64_t(s.P) * s.B * a.Lp;
    const uint64_t row_elems = uint64_t(s.H) * s.d_h;
    const uint64_t run_elems = row_elems / uint64_t(G);
    const uint64_t total = rows * row_elems;
    if (total == 0) return ULYSSES_OK;
    const int sms = device_sm_count();
    constexpr int kThreads = 256;
    const bool vec_ok = (run_elems % 8 == 0) && row_elems <= 8 * 512 && total / 8 < (1ull << 32) &&
                        ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) % 16 == 0);
    if (vec_ok) {
        a.rows = static_cast<uint32_t>(rows);
        a.row_vecs = static_cast<uint32_t>(row_elems / 8);
        a.run_vecs = static_cast<uint32_t>(run_elems / 8);
        const uint32_t vpl = (a.row_vecs + 31) / 32;
        const int unroll = vpl <= 2 ? 8 : vpl <= 4 ? 4 : vpl <= 8 ? 2 : 1;
        const uint64_t rows_per_cta = uint64_t(kThreads / 32) * unroll;
        uint64_t blocks = (rows + rows_per_cta - 1) / rows_per_cta;
        const uint64_t cap = uint64_t(sms) * 2;
        if (blocks > cap) blocks = cap;
        const unsigned nb = unsigned(blocks);
        if (vpl <= 1) relayout_row_kernel<1, 8><<<nb, kThreads, 0, stream>>>(a);
        else if (vpl <= 2) relayout_row_kernel<2, 8><<<nb, kThreads, 0, stream>>>(a);
        else if (vpl <= 4) relayout_row_kernel<4, 4><<<nb, kThreads, 0, stream>>>(a);
        else if (vpl <= 8) relayout_row_kernel<8, 2><<<nb, kThreads, 0, stream>>>(a);
        else relayout_row_kernel<16, 1><<<nb, kThreads, 0, stream>>>(a);
    } else {
        RelayoutArgs e = a;
        uint64_t blocks = (total + kThreads - 1) / kThreads;
        const uint64_t cap = uint64_t(sms) * 16;
        if (blocks > cap) blocks = cap;
        relayout_elem_kernel<<<unsigned(blocks), kThreads, 0, stream>>>(e, total);
    }
    return cudaGetLastError() == cudaSuccess ? ULYSSES_OK : ULYSSES_ERR_CUDA;
}

// ---------------------------------------------------------------------------------------
// Key/value relayouts with replicated heads (P > Hkv): head group g holds one key/value
// head, g / rep with rep = P / Hkv (head-sharded [P][B][L][1][d]).
//   seq->head: every destination row copies its source head's d elements;
//   head->seq: every key/value head receives the fp32 sum of its rep copies (ascending g),
//              rounded to bf16 (the adjoint, for gradients).
// One thread per VEC consecutive elements of a destination row.
// ---------------------------------------------------------------------------------------
struct KvRepArgs {
    const void* in;
    void* out;
    uint64_t P, B, L, Lp, Hkv, d, rep;
};

template <int VEC>
__global__ void __launch_bounds__(256) kv_rep_to_head_kernel(KvRepArgs a, uint64_t total) {
    using T = typename std::conditional<VEC == 8, uint4, uint16_t>::type;
    const T* in = static_cast<const T*>(a.in);
    T* out = static_cast<T*>(a.out);
    const uint64_t dv = a.d / VEC;
    for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += uint64_t(gridDim.x) * blockDim.x) {
        // destination [g][b][s][v]
        const uint64_t v = i % dv;
        const uint64_t row = i / dv;
        const uint64_t s = row % a.L;
        const uint64_t gb = row / a.L;
        const uint64_t b = gb % a.B;
        const uint64_t g = gb / a.B;
        const uint64_t h = g / a.rep;
        const uint64_t src = (((s / a.Lp) * a.B + b) * a.Lp + s % a.Lp) * a.Hkv + h;
        out[i] = in[src * dv + v];
    }
}

template <int VEC>
__global__ void __launch_bounds__(256) kv_rep_to_seq_sum_kernel(KvRepArgs a, uint64_t total) {
    const __nv_bfloat16* in = static_cast<const __nv_bfloat16*>(a.in);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    const uint64_t dv = a.d / VEC;
    for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += uint64_t(gridDim.x) * blockDim.x) {
        // destination [r][b][t][h][v]
        const uint64_t v = i % dv;
        const uint64_t row = i / dv;
        const uint64_t h = row % a.Hkv;
        const uint64_t tok = row / a.Hkv;  // (r * B + b) * Lp + t
        const uint64_t t = tok % a.Lp;
        const uint64_t rb = tok / a.Lp;
        const uint64_t b = rb % a.B;
        const uint64_t r = rb / a.B;
        const uint64_t s = r * a.Lp + t;
        float acc[VEC];
#pragma unroll
        for (int x = 0; x < VEC; ++x) acc[x] = 0.f;
        for (uint64_t g = h * a.rep; g < (h + 1) * a.rep; ++g) {
            const __nv_bfloat16* src = in + ((g * a.B + b) * a.L + s) * a.d + v * VEC;
            if (VEC == 8) {
                const uint4 w = *reinterpret_cast<const uint4*>(src);
                const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
                for (int x = 0; x < VEC / 2; ++x) {
                    const float2 f = __bfloat1622float2(w2[x]);
                    acc[2 * x] += f.x;
                    acc[2 * x + 1] += f.y;
                }
            } else {
#pragma unroll
                for (int x = 0; x < VEC; ++x) acc[x] += __bfloat162float(src[x]);
            }
        }
        __nv_bfloat16* dst = out + i * VEC;
        if (VEC == 8) {
            uint4 w;
            w.x = pack_bf16(acc[0], acc[1]);
            w.y = pack_bf16(acc[2], acc[3]);
            w.z = pack_bf16(acc[4], acc[5]);
            w.w = pack_bf16(acc[6], acc[7]);
            *reinterpret_cast<uint4*>(dst) = w;
        } else {
#pragma unroll
            for (int x = 0; x < VEC; ++x) dst[x] = __float2bfloat16_rn(acc[x]);
        }
    }
}

int launch_kv_replicated(const ulysses_shape_t& s, const void* in, void* out, cudaStream_t stream, bool to_head) {
    KvRepArgs a{};
    a.in = in;
    a.out = out;
    a.P = uint64_t(s.P); a.B = uint64_t(s.B); a.L = uint64_t(s.L); a.Lp = a.L / a.P;
    a.Hkv = uint64_t(s.H_kv); a.d = uint64_t(s.d_h); a.rep = a.P / a.Hkv;
    const bool vec = (a.d % 8 == 0) && ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) % 16 == 0);
    const uint64_t elems = to_head ? a.P * a.B * a.L * a.d : a.P * a.B * a.Lp * a.Hkv * a.d;
    const uint64_t total = elems / (vec ? 8 : 1);
    if (total == 0) return ULYSSES_OK;
    uint64_t blocks = (total + 255) / 256;
    const uint64_t cap = uint64_t(device_sm_count()) * 16;
    if (blocks > cap) blocks = cap;
    if (to_head) {
        if (vec) kv_rep_to_head_kernel<8><<<unsigned(blocks), 256, 0, stream>>>(a, total);
        else kv_rep_to_head_kernel<1><<<unsigned(blocks), 256, 0, stream>>>(a, total);
    } else {
        if (vec) kv_rep_to_seq_sum_kernel<8><<<unsigned(blocks), 256, 0, stream>>>(a, total);
        else kv_rep_to_seq_sum_kernel<1><<<unsigned(blocks), 256, 0, stream>>>(a, total);
    }
    return cudaGetLastError() == cudaSuccess ? ULYSSES_OK : ULYSSES_ERR_CUDA;
}

}  // namespace ulysses
