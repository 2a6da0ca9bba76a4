// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ulysses.h"

namespace ulysses {

constexpr int kTile = 128;      // query / key tile edge of the attention kernels
constexpr int kBwdQTile = 64;   // query rows per step of the backward kernel

int device_sm_count();
// Raises kernel fn's dynamic shared-memory limit to `bytes` on the current device, once per
// (kernel, device): thread-safe, and a failed attempt is retried by the next call.
bool set_max_dynamic_smem(const void* fn, int bytes);
uint32_t* device_error_word();  // device address of this device's error word (nullptr on failure)

// Key/value head arrangement of a shape (grouped-query attention when Hkv < H).
struct KvInfo {
    int Hkv;   // key/value heads
    int G;     // query heads per key/value head, H / Hkv
    int Hkvp;  // key/value heads per head group in the head-sharded layout
    int rep;   // head groups holding a copy of each key/value head (1 unless P > Hkv)
};
inline int shape_hkv(const ulysses_shape_t& s) { return s.H_kv > 0 ? s.H_kv : s.H; }
inline KvInfo kv_info(const ulysses_shape_t& s) {
    KvInfo k{};
    k.Hkv = shape_hkv(s);
    k.G = s.H / k.Hkv;
    if (k.Hkv % s.P == 0) { k.Hkvp = k.Hkv / s.P; k.rep = 1; }
    else { k.Hkvp = 1; k.rep = s.P / k.Hkv; }
    return k;
}

// cuTensorMapEncodeTiled (looked up at run time) with the 128-byte swizzle, 256-byte L2
// promotion and zero fill out of bounds.
bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, const void* base,
                       const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                       const cuuint32_t* elem_strides);

// Encodes a 5-D bf16 tensor map over (d, head, row, batch, unit) with a box of
// (64, 1, box_rows, 1, 1), 128-byte swizzle and zero fill out of bounds, for a tensor with
// `heads` heads in the token layout and `group_heads` per head group in the head layout:
//   token layout: dims (d, heads, Lp, B, P);  head layout: dims (d, group_heads, L, B, P).
bool encode_qkv_map(CUtensorMap* map, const void* base, const ulysses_shape_t& s, int layout, int box_rows,
                    int heads, int group_heads);

struct MaskArgs {
    int kind;
    const int32_t* q_rowptr;
    const int32_t* q_kcols;
    const int32_t* k_colptr;
    const int32_t* k_qrows;
};

// The token <-> head relayouts over P shards and G head groups (G <= 0: G = P). With P = 1 and
// G > 1 it packs one rank's token shard into G per-destination chunks (or unpacks them).
int launch_relayout(const ulysses_shape_t& s, const void* in, void* out, cudaStream_t stream, bool to_head,
                    int G = 0);
// Key/value relayouts with replication (P > Hkv): seq->head copies, head->seq sums the copies.
int launch_kv_replicated(const ulysses_shape_t& s, const void* in, void* out, cudaStream_t stream, bool to_head);

// How one forward launch joins a chain of launches over the same query rows (the block pairs of
// the Ulysses-ring hybrid). The default is a standalone forward.
struct FwdChain {
    // 0 write O (bf16) and lse; 1 store this launch's normalised O and lse to the fp32 running
    // pair; 2 merge into the running pair (online-softmax rule); 3 merge and write O and lse
    int mode = 0;
    float* o_acc = nullptr;    // same layout as O, fp32
    float* lse_acc = nullptr;  // same layout as lse
};

int launch_attn_fwd(const ulysses_shape_t& s, const MaskArgs& m, float scale, int layout, const void* q,
                    const void* k, const void* v, void* o, float* lse, cudaStream_t stream,
                    const FwdChain& chain = FwdChain());

// How one backward launch joins a chain of launches that add into the same gradients (the block
// pairs of the Ulysses-ring hybrid). The default is a standalone backward.
struct BwdChain {
    bool prep = true;     // compute Delta and zero the fp32 dQ accumulator (a query block's first launch)
    bool convert = true;  // write dQ from the accumulator (a query block's last launch)
    // dK, dV: 0 stored bf16; 1 stored fp32 to the accumulators; 2 added into them;
    // 3 stored bf16(accumulator + this launch's part)
    int dkv_mode = 0;
    float* dk_acc = nullptr;  // same layout as dK, fp32
    float* dv_acc = nullptr;
};

int launch_attn_bwd(const ulysses_shape_t& s, const MaskArgs& m, float scale, int layout, const void* q,
                    const void* k, const void* v, const void* o, const float* lse, const void* dO, void* dq,
                    void* dk, void* dv, void* workspace, cudaStream_t stream, const BwdChain& chain = BwdChain());

size_t bwd_workspace_bytes(const ulysses_shape_t& s);

// Ulysses-ring hybrid over P_ring ring blocks (P_ring <= kMaxRing)
constexpr int kMaxRing = 64;
size_t usp_workspace_bytes(const ulysses_shape_t& s, int P_ring);
// Waits for and destroys the calling thread's side streams and their events (USP forward).
bool release_side_streams();
int launch_usp_fwd(const ulysses_shape_t& s, int P_ring, const MaskArgs& m, float scale, const void* q, const void* k,
                   const void* v, void* o, float* lse, void* ws, cudaStream_t stream);
int launch_usp_bwd(const ulysses_shape_t& s, int P_ring, const MaskArgs& m, float scale, const void* q, const void* k,
                   const void* v, const void* o, const float* lse, const void* dO, void* dq, void* dk, void* dv,
                   void* ws, cudaStream_t stream);

// C[M][N] = A[M][K] B[N][K]^T in bf16 (fp32 accumulation); column range [col0[i], col0[i+1])
// of C is written row-major to out[i] with row pitch ld[i].
int launch_proj_gemm(int M, int N, int K, const void* a, const void* b, int n_out, const int* col0, void* const* out,
                     const int* ld, cudaStream_t stream);

inline int gcd_int(int a, int b) {
    while (b) { int t = a % b; a = b; b = t; }
    return a;
}

}  // namespace ulysses
