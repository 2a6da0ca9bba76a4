// Host side of the C ABI declared in include/ulysses.h: argument validation, tensor-map
// encoding, the per-device error word and the block-sparse tile-list builder.
#include <cstring>
#include <mutex>
#include <set>
#include <utility>
#include <vector>

#include "common.cuh"
#include "ulysses_internal.h"

namespace ulysses {

// The per-process error word of each device that loads this library (4 bytes).
__device__ uint32_t g_error_word_storage;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices] = {};
uint32_t* g_err[kMaxDevices] = {};
// signature of cuTensorMapEncodeTiled (driver API), looked up at run time
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

bool load_encode_fn() {
    if (g_encode) return true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return false;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int device_sm_count() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return 148;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sms[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

bool set_max_dynamic_smem(const void* fn, int bytes) {
    const int dev = current_device();
    if (dev < 0) return false;
    static std::mutex mu;
    static std::set<std::pair<const void*, int>> done;
    std::lock_guard<std::mutex> lk(mu);
    if (done.count({fn, dev})) return true;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
    done.insert({fn, dev});
    return true;
}

uint32_t* device_error_word() {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_error_word_storage) != cudaSuccess) return nullptr;
        g_err[dev] = static_cast<uint32_t*>(ptr);
    }
    return g_err[dev];
}

namespace {

// A tensor map is a pure function of its arguments (the address, not the memory behind it), so
// each host thread keeps the maps it encoded most recently and hands out a copy when the same
// arguments come again: 64 slots, direct-mapped by a hash of the arguments.
struct MapKey {
    uint64_t dtype, rank;
    uint64_t base;
    cuuint64_t dims[5], strides[4];
    cuuint32_t box[5], estr[5];
};
struct MapSlot {
    MapKey key;
    CUtensorMap map;
    bool valid;
};
thread_local MapSlot t_maps[64];

bool encode_memo(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, const void* base, const cuuint64_t* dims,
                 const cuuint64_t* strides, const cuuint32_t* box, const cuuint32_t* estr) {
    if (rank == 0 || rank > 5) return false;
    MapKey k;
    std::memset(&k, 0, sizeof(k));
    k.dtype = uint64_t(dtype);
    k.rank = rank;
    k.base = reinterpret_cast<uintptr_t>(base);
    for (uint32_t i = 0; i < rank; ++i) {
        k.dims[i] = dims[i];
        k.box[i] = box[i];
        k.estr[i] = estr[i];
        if (i + 1 < rank) k.strides[i] = strides[i];
    }
    uint64_t h = 1469598103934665603ull;  // FNV-1a over the key's bytes
    const unsigned char* kb = reinterpret_cast<const unsigned char*>(&k);
    for (size_t i = 0; i < sizeof(k); ++i) h = (h ^ kb[i]) * 1099511628211ull;
    MapSlot& sl = t_maps[(h ^ (h >> 32)) & 63];
    if (sl.valid && std::memcmp(&sl.key, &k, sizeof(k)) == 0) {
        *map = sl.map;
        return true;
    }
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!load_encode_fn()) return false;
    }
    if (g_encode(map, dtype, rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    sl.key = k;
    sl.map = *map;
    sl.valid = true;
    return true;
}

}  // namespace

bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, const void* base,
                       const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                       const cuuint32_t* elem_strides) {
    return encode_memo(map, dtype, rank, base, dims, strides, box, elem_strides);
}

bool encode_qkv_map(CUtensorMap* map, const void* base, const ulysses_shape_t& s, int layout, int box_rows,
                    int heads, int group_heads) {
    const uint64_t d = s.d_h, H = heads, P = s.P, B = s.B, L = s.L;
    const uint64_t Hp = group_heads, Lp = L / P;
    cuuint64_t dims[5];
    cuuint64_t strides[4];  // bytes, dims 1..4
    if (layout == ULYSSES_LAYOUT_TOKEN_SHARDED) {
        dims[0] = d; dims[1] = H; dims[2] = Lp; dims[3] = B; dims[4] = P;
    } else {
        dims[0] = d; dims[1] = Hp; dims[2] = L; dims[3] = B; dims[4] = P;
    }
    strides[0] = dims[0] * 2;
    strides[1] = strides[0] * dims[1];
    strides[2] = strides[1] * dims[2];
    strides[3] = strides[2] * dims[3];
    cuuint32_t box[5] = {64, 1, static_cast<cuuint32_t>(box_rows), 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return encode_memo(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, strides, box, estr);
}

namespace {

int validate_shape(const ulysses_shape_t& s) {
    if (s.B < 0 || s.L < 0 || s.H <= 0 || s.d_h <= 0 || s.P <= 0 || s.H_kv < 0) return ULYSSES_ERR_INVALID_ARG;
    if (s.H % s.P != 0 || s.L % s.P != 0) return ULYSSES_ERR_INVALID_ARG;
    // grouped key/value heads: whole groups of query heads, and whole (or replicated) heads per group
    const int hkv = shape_hkv(s);
    if (s.H % hkv != 0 || (hkv % s.P != 0 && s.P % hkv != 0)) return ULYSSES_ERR_INVALID_ARG;
    // element counts must fit the kernels' 64-bit offsets and 32-bit row counters
    if (uint64_t(s.B) * uint64_t(s.L) * uint64_t(s.H) * uint64_t(s.d_h) > (1ull << 40)) return ULYSSES_ERR_INVALID_ARG;
    return ULYSSES_OK;
}

int validate_attn(const ulysses_shape_t& s, const ulysses_mask_t* mask, int layout) {
    int rc = validate_shape(s);
    if (rc != ULYSSES_OK) return rc;
    if (!mask) return ULYSSES_ERR_INVALID_ARG;
    if (mask->kind != ULYSSES_MASK_NONE && mask->kind != ULYSSES_MASK_CAUSAL && mask->kind != ULYSSES_MASK_BLOCK_SPARSE)
        return ULYSSES_ERR_INVALID_ARG;
    if (layout != ULYSSES_LAYOUT_TOKEN_SHARDED && layout != ULYSSES_LAYOUT_HEAD_SHARDED) return ULYSSES_ERR_INVALID_ARG;
    if (mask->kind == ULYSSES_MASK_BLOCK_SPARSE) {
        if (mask->tile != kTile) return ULYSSES_ERR_UNSUPPORTED;
        if (!mask->q_rowptr || !mask->q_kcols || !mask->k_colptr || !mask->k_qrows || mask->nnz < 0)
            return ULYSSES_ERR_INVALID_ARG;
    }
    if (s.d_h != 64 && s.d_h != 128) return ULYSSES_ERR_UNSUPPORTED;
    if (layout == ULYSSES_LAYOUT_TOKEN_SHARDED && (s.L / s.P) % 8 != 0 && s.L > 0) return ULYSSES_ERR_UNSUPPORTED;
    // grid limits: tiles along x, B*H along y
    if (uint64_t(s.B) * s.H > 65535) return ULYSSES_ERR_UNSUPPORTED;
    return ULYSSES_OK;
}

float resolve_scale(float scale, int d) { return scale > 0.f ? scale : 1.0f / sqrtf(float(d)); }

}  // namespace

// Two warps wait on an mbarrier that nothing ever arrives on, through the same bounded wait
// the attention kernels use: the first to run out of time records the error word and sets
// the CTA's abort flag, the other sees the flag (or runs out too), and both return.
__global__ void selftest_timeout_kernel(uint32_t* err) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const Abort ab{&abort_flag, err, KID_SELFTEST};
    if ((threadIdx.x & 31) == 0) mbar_wait(&bar, 0, ab, ROLE_SELFTEST, 1 + threadIdx.x / 32);
    __syncwarp();
    __syncthreads();
}

}  // namespace ulysses

using namespace ulysses;

extern "C" {

const char* ulysses_status_string(int status) {
    switch (status) {
        case ULYSSES_OK: return "ULYSSES_OK";
        case ULYSSES_ERR_INVALID_ARG: return "ULYSSES_ERR_INVALID_ARG";
        case ULYSSES_ERR_UNSUPPORTED: return "ULYSSES_ERR_UNSUPPORTED";
        case ULYSSES_ERR_MISALIGNED: return "ULYSSES_ERR_MISALIGNED";
        case ULYSSES_ERR_CUDA: return "ULYSSES_ERR_CUDA";
        case ULYSSES_ERR_DEVICE_TIMEOUT: return "ULYSSES_ERR_DEVICE_TIMEOUT";
        default: return "ULYSSES_ERR_UNKNOWN";
    }
}

static int relayout_common(ulysses_shape_t shape, const void* in, void* out, void* stream, bool to_head) {
    int rc = validate_shape(shape);
    if (rc != ULYSSES_OK) return rc;
    const uint64_t n = uint64_t(shape.B) * shape.L * shape.H * shape.d_h;
    if (n == 0) return ULYSSES_OK;
    if (!in || !out) return ULYSSES_ERR_INVALID_ARG;
    if (in == out) return ULYSSES_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) & 1u) return ULYSSES_ERR_MISALIGNED;
    return launch_relayout(shape, in, out, static_cast<cudaStream_t>(stream), to_head);
}

int ulysses_seq_to_head(ulysses_shape_t shape, const void* in, void* out, void* stream) {
    return relayout_common(shape, in, out, stream, true);
}

int ulysses_head_to_seq(ulysses_shape_t shape, const void* in, void* out, void* stream) {
    return relayout_common(shape, in, out, stream, false);
}

// One process's side of the all-to-alls when the P ranks are P processes: its token shard
// [B][L/P][H][d] split into P contiguous per-destination chunks [P][B][L/P][H/P][d] (pack),
// and the inverse (unpack). Only B, L, H, d_h and P take part; H is the tensor's own head
// count (H_kv for keys and values), so H_kv is ignored.
static int a2a_common(ulysses_shape_t shape, const void* in, void* out, void* stream, bool pack) {
    if (shape.B < 0 || shape.L < 0 || shape.H <= 0 || shape.d_h <= 0 || shape.P <= 0) return ULYSSES_ERR_INVALID_ARG;
    if (shape.H % shape.P != 0 || shape.L % shape.P != 0) return ULYSSES_ERR_INVALID_ARG;
    if (uint64_t(shape.B) * uint64_t(shape.L) * uint64_t(shape.H) * uint64_t(shape.d_h) > (1ull << 40))
        return ULYSSES_ERR_INVALID_ARG;
    const uint64_t n = uint64_t(shape.B) * (shape.L / shape.P) * shape.H * shape.d_h;
    if (n == 0) return ULYSSES_OK;
    if (!in || !out) return ULYSSES_ERR_INVALID_ARG;
    if (in == out) return ULYSSES_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) & 1u) return ULYSSES_ERR_MISALIGNED;
    // one shard (P = 1) of L / P tokens, split into P head groups
    ulysses_shape_t one = shape;
    one.L = shape.L / shape.P;
    one.P = 1;
    one.H_kv = 0;
    return launch_relayout(one, in, out, static_cast<cudaStream_t>(stream), pack, shape.P);
}

int ulysses_a2a_pack(ulysses_shape_t shape, const void* in, void* out, void* stream) {
    return a2a_common(shape, in, out, stream, true);
}

int ulysses_a2a_unpack(ulysses_shape_t shape, const void* in, void* out, void* stream) {
    return a2a_common(shape, in, out, stream, false);
}

// Key/value relayouts: without replication they are the plain relayouts of a tensor with
// H_kv heads; with it (P > H_kv) a dedicated kernel copies (seq->head) or sums (head->seq).
static int kv_relayout_common(ulysses_shape_t shape, const void* in, void* out, void* stream, bool to_head) {
    // only B, L, d_h, P and the key/value head count take part (H only when H_kv is 0)
    const int hkv = shape_hkv(shape);
    if (shape.B < 0 || shape.L < 0 || shape.d_h <= 0 || shape.P <= 0 || hkv <= 0 || shape.L % shape.P != 0 ||
        (hkv % shape.P != 0 && shape.P % hkv != 0))
        return ULYSSES_ERR_INVALID_ARG;
    if (uint64_t(shape.B) * uint64_t(shape.L) * uint64_t(hkv) * uint64_t(shape.d_h) > (1ull << 40))
        return ULYSSES_ERR_INVALID_ARG;
    const KvInfo kv = kv_info(shape);
    if (uint64_t(shape.B) * shape.L * kv.Hkv * shape.d_h == 0) return ULYSSES_OK;
    if (!in || !out) return ULYSSES_ERR_INVALID_ARG;
    if (in == out) return ULYSSES_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) & 1u) return ULYSSES_ERR_MISALIGNED;
    ulysses_shape_t s = shape;
    s.H = kv.Hkv;
    s.H_kv = kv.Hkv;
    if (kv.rep == 1) return launch_relayout(s, in, out, static_cast<cudaStream_t>(stream), to_head);
    return launch_kv_replicated(s, in, out, static_cast<cudaStream_t>(stream), to_head);
}

int ulysses_kv_seq_to_head(ulysses_shape_t shape, const void* in, void* out, void* stream) {
    return kv_relayout_common(shape, in, out, stream, true);
}

int ulysses_kv_head_to_seq_sum(ulysses_shape_t shape, const void* in, void* out, void* stream) {
    return kv_relayout_common(shape, in, out, stream, false);
}

// Projections: C[M][N] = A[M][K] B[N][K]^T over the M = B * L token rows of the token-sharded
// layout. TMA needs 16-byte row pitches (K % 8 == 0); the epilogue routes 32-column chunks.
static int validate_proj(const ulysses_shape_t& s, int hidden) {
    int rc = validate_shape(s);
    if (rc != ULYSSES_OK) return rc;
    if (hidden <= 0) return ULYSSES_ERR_INVALID_ARG;
    if (hidden % 32 != 0 || (s.H * s.d_h) % 32 != 0 || (shape_hkv(s) * s.d_h) % 32 != 0) return ULYSSES_ERR_UNSUPPORTED;
    if (uint64_t(s.B) * s.L > 0x7fffffffull) return ULYSSES_ERR_UNSUPPORTED;
    return ULYSSES_OK;
}

int ulysses_qkv_proj(ulysses_shape_t shape, int hidden, const void* x, const void* w_qkv, void* q, void* k, void* v,
                     void* stream) {
    int rc = validate_proj(shape, hidden);
    if (rc != ULYSSES_OK) return rc;
    const int M = shape.B * shape.L;
    if (M == 0) return ULYSSES_OK;
    if (!x || !w_qkv || !q || !k || !v) return ULYSSES_ERR_INVALID_ARG;
    const void* ins[] = {x, w_qkv};
    const void* outs[] = {q, k, v};
    for (const void* a : outs)
        for (const void* b : ins)
            if (a == b) return ULYSSES_ERR_INVALID_ARG;
    if (q == k || q == v || k == v) return ULYSSES_ERR_INVALID_ARG;
    for (const void* a : ins)
        if (!aligned16(a)) return ULYSSES_ERR_MISALIGNED;
    for (const void* a : outs)
        if (!aligned16(a)) return ULYSSES_ERR_MISALIGNED;
    const int hq = shape.H * shape.d_h, hkv = shape_hkv(shape) * shape.d_h;
    const int col0[4] = {0, hq, hq + hkv, hq + 2 * hkv};
    void* out[3] = {q, k, v};
    const int ld[3] = {hq, hkv, hkv};
    return launch_proj_gemm(M, hq + 2 * hkv, hidden, x, w_qkv, 3, col0, out, ld, static_cast<cudaStream_t>(stream));
}

int ulysses_out_proj(ulysses_shape_t shape, int hidden, const void* o, const void* w_o, void* y, void* stream) {
    int rc = validate_proj(shape, hidden);
    if (rc != ULYSSES_OK) return rc;
    const int M = shape.B * shape.L;
    if (M == 0) return ULYSSES_OK;
    if (!o || !w_o || !y) return ULYSSES_ERR_INVALID_ARG;
    if (y == o || y == w_o) return ULYSSES_ERR_INVALID_ARG;
    if (!aligned16(o) || !aligned16(w_o) || !aligned16(y)) return ULYSSES_ERR_MISALIGNED;
    const int col0[2] = {0, hidden};
    void* out[1] = {y};
    const int ld[1] = {hidden};
    return launch_proj_gemm(M, hidden, shape.H * shape.d_h, o, w_o, 1, col0, out, ld, static_cast<cudaStream_t>(stream));
}

// Ulysses-ring hybrid: the full shape only needs L % P == 0 and P % P_ring == 0; each ring block
// (L / P_ring tokens, P / P_ring shards) must be a valid token-sharded attention shape.
static int validate_usp(const ulysses_shape_t& s, int P_ring, const ulysses_mask_t* mask) {
    if (s.B < 0 || s.L < 0 || s.H <= 0 || s.d_h <= 0 || s.P <= 0 || s.H_kv < 0) return ULYSSES_ERR_INVALID_ARG;
    if (P_ring <= 0 || P_ring > kMaxRing || s.P % P_ring != 0 || s.L % s.P != 0) return ULYSSES_ERR_INVALID_ARG;
    if (!mask) return ULYSSES_ERR_INVALID_ARG;
    if (mask->kind == ULYSSES_MASK_BLOCK_SPARSE) return ULYSSES_ERR_UNSUPPORTED;
    ulysses_shape_t sub = s;
    sub.L = s.L / P_ring;
    sub.P = s.P / P_ring;
    return validate_attn(sub, mask, ULYSSES_LAYOUT_TOKEN_SHARDED);
}

size_t ulysses_usp_workspace_size(ulysses_shape_t shape, int P_ring) {
    ulysses_mask_t causal{ULYSSES_MASK_CAUSAL, kTile, nullptr, nullptr, nullptr, nullptr, 0};
    if (validate_usp(shape, P_ring, &causal) != ULYSSES_OK) return 0;
    return usp_workspace_bytes(shape, P_ring);
}

int ulysses_usp_attn_fwd(ulysses_shape_t shape, int P_ring, const ulysses_mask_t* mask, float softmax_scale,
                         const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                         size_t workspace_bytes, void* stream) {
    int rc = validate_usp(shape, P_ring, mask);
    if (rc != ULYSSES_OK) return rc;
    if (shape.B == 0 || shape.L == 0) return ULYSSES_OK;
    if (!q || !k || !v || !o || !lse || !workspace) return ULYSSES_ERR_INVALID_ARG;
    if (o == q || o == k || o == v) return ULYSSES_ERR_INVALID_ARG;
    if (workspace_bytes < usp_workspace_bytes(shape, P_ring)) return ULYSSES_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return ULYSSES_ERR_MISALIGNED;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ULYSSES_ERR_MISALIGNED;
    MaskArgs m{mask->kind, nullptr, nullptr, nullptr, nullptr};
    return launch_usp_fwd(shape, P_ring, m, resolve_scale(softmax_scale, shape.d_h), q, k, v, o, lse, workspace,
                          static_cast<cudaStream_t>(stream));
}

int ulysses_usp_attn_bwd(ulysses_shape_t shape, int P_ring, const ulysses_mask_t* mask, float softmax_scale,
                         const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                         void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = validate_usp(shape, P_ring, mask);
    if (rc != ULYSSES_OK) return rc;
    if (shape.B == 0 || shape.L == 0) return ULYSSES_OK;
    if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv || !workspace) return ULYSSES_ERR_INVALID_ARG;
    if (workspace_bytes < usp_workspace_bytes(shape, P_ring)) return ULYSSES_ERR_INVALID_ARG;
    const void* ins[] = {q, k, v, o, lse, dO};
    const void* outs[] = {dq, dk, dv, workspace};
    for (const void* a : outs)
        for (const void* b : ins)
            if (a == b) return ULYSSES_ERR_INVALID_ARG;
    if (dq == dk || dq == dv || dk == dv) return ULYSSES_ERR_INVALID_ARG;
    for (const void* a : ins)
        if (!aligned16(a)) return ULYSSES_ERR_MISALIGNED;
    for (const void* a : outs)
        if (!aligned16(a)) return ULYSSES_ERR_MISALIGNED;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ULYSSES_ERR_MISALIGNED;
    MaskArgs m{mask->kind, nullptr, nullptr, nullptr, nullptr};
    return launch_usp_bwd(shape, P_ring, m, resolve_scale(softmax_scale, shape.d_h), q, k, v, o, lse, dO, dq, dk, dv,
                          workspace, static_cast<cudaStream_t>(stream));
}

int ulysses_attn_fwd(ulysses_shape_t shape, const ulysses_mask_t* mask, float softmax_scale, int io_layout,
                     const void* q, const void* k, const void* v, void* o, float* lse, void* stream) {
    int rc = validate_attn(shape, mask, io_layout);
    if (rc != ULYSSES_OK) return rc;
    if (shape.B == 0 || shape.L == 0) return ULYSSES_OK;
    if (!q || !k || !v || !o || !lse) return ULYSSES_ERR_INVALID_ARG;
    if (o == q || o == k || o == v) return ULYSSES_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return ULYSSES_ERR_MISALIGNED;
    MaskArgs m{mask->kind, mask->q_rowptr, mask->q_kcols, mask->k_colptr, mask->k_qrows};
    return launch_attn_fwd(shape, m, resolve_scale(softmax_scale, shape.d_h), io_layout, q, k, v, o, lse,
                           static_cast<cudaStream_t>(stream));
}

size_t ulysses_attn_bwd_workspace_size(ulysses_shape_t shape) {
    if (validate_shape(shape) != ULYSSES_OK) return 0;
    return bwd_workspace_bytes(shape);
}

int ulysses_attn_bwd(ulysses_shape_t shape, const ulysses_mask_t* mask, float softmax_scale, int io_layout,
                     const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                     void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, void* stream) {
    int rc = validate_attn(shape, mask, io_layout);
    if (rc != ULYSSES_OK) return rc;
    if (shape.B == 0 || shape.L == 0) return ULYSSES_OK;
    if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv || !workspace) return ULYSSES_ERR_INVALID_ARG;
    if (workspace_bytes < bwd_workspace_bytes(shape)) return ULYSSES_ERR_INVALID_ARG;
    const void* ins[] = {q, k, v, o, lse, dO};
    const void* outs[] = {dq, dk, dv, workspace};
    for (const void* a : outs)
        for (const void* b : ins)
            if (a == b) return ULYSSES_ERR_INVALID_ARG;
    if (dq == dk || dq == dv || dk == dv) return ULYSSES_ERR_INVALID_ARG;
    for (const void* a : ins)
        if (!aligned16(a)) return ULYSSES_ERR_MISALIGNED;
    for (const void* a : outs)
        if (!aligned16(a)) return ULYSSES_ERR_MISALIGNED;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ULYSSES_ERR_MISALIGNED;
    MaskArgs m{mask->kind, mask->q_rowptr, mask->q_kcols, mask->k_colptr, mask->k_qrows};
    return launch_attn_bwd(shape, m, resolve_scale(softmax_scale, shape.d_h), io_layout, q, k, v, o, lse, dO, dq, dk,
                           dv, workspace, static_cast<cudaStream_t>(stream));
}

int ulysses_bsmask_build_window_global(int L, int tile, int window_before, int window_after, int global_stride,
                                       int32_t* rowptr, int32_t* kcols, int32_t* colptr, int32_t* qrows, int* nnz) {
    if (L <= 0 || tile <= 0 || window_before < 0 || window_after < 0 || !nnz || !rowptr || !colptr)
        return ULYSSES_ERR_INVALID_ARG;
    const int n = (L + tile - 1) / tile;
    // pass 1: count, building CSR; a key tile is active for query tile qt if it lies in the
    // window [qt - window_before, qt + window_after] or is a global tile
    std::vector<int32_t> rp(n + 1, 0), cols;
    cols.reserve(size_t(n) * (window_before + window_after + 1 + (global_stride > 0 ? n / global_stride + 1 : 0)));
    for (int qt = 0; qt < n; ++qt) {
        const int lo = qt - window_before < 0 ? 0 : qt - window_before;
        const int hi = qt + window_after > n - 1 ? n - 1 : qt + window_after;
        for (int kt = 0; kt < n; ++kt) {
            const bool win = kt >= lo && kt <= hi;
            const bool glob = global_stride > 0 && kt % global_stride == 0;
            if (win || glob) cols.push_back(kt);
        }
        rp[qt + 1] = int32_t(cols.size());
    }
    const int total = int(cols.size());
    const int cap = *nnz;
    *nnz = total;
    if (cap < total || !kcols || !qrows) return ULYSSES_ERR_INVALID_ARG;
    std::memcpy(rowptr, rp.data(), sizeof(int32_t) * (n + 1));
    std::memcpy(kcols, cols.data(), sizeof(int32_t) * total);
    // CSC by counting sort over key tiles; query tiles come out ascending
    std::vector<int32_t> cnt(n + 1, 0);
    for (int e = 0; e < total; ++e) cnt[cols[e] + 1]++;
    for (int kt = 0; kt < n; ++kt) cnt[kt + 1] += cnt[kt];
    std::memcpy(colptr, cnt.data(), sizeof(int32_t) * (n + 1));
    std::vector<int32_t> pos(cnt.begin(), cnt.end() - 1);
    for (int qt = 0; qt < n; ++qt)
        for (int e = rp[qt]; e < rp[qt + 1]; ++e) qrows[pos[cols[e]]++] = qt;
    return ULYSSES_OK;
}

int ulysses_selftest_timeout(void* stream) {
    uint32_t* err = device_error_word();
    if (!err) return ULYSSES_ERR_CUDA;
    selftest_timeout_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(err);
    return cudaGetLastError() == cudaSuccess ? ULYSSES_OK : ULYSSES_ERR_CUDA;
}

int ulysses_get_device_status(void* stream, uint32_t* detail) {
    uint32_t* err = device_error_word();
    if (!err) return ULYSSES_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return ULYSSES_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpyFromSymbol(&word, g_error_word_storage, sizeof(word)) != cudaSuccess) return ULYSSES_ERR_CUDA;
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_error_word_storage, &zero, sizeof(zero)) != cudaSuccess) return ULYSSES_ERR_CUDA;
    if (detail) *detail = word;
    return word == 0 ? ULYSSES_OK : ULYSSES_ERR_DEVICE_TIMEOUT;
}

int ulysses_shutdown(void) {
    for (MapSlot& sl : t_maps) sl.valid = false;
    return release_side_streams() ? ULYSSES_OK : ULYSSES_ERR_CUDA;
}

}  // extern "C"
