// spark_attn.cu -- host side of the C ABI declared in include/spark_attn.h:
// argument validation, RoPE frequency tables, TMA tensor maps, work planning
// and the kernel launches.  No device memory is allocated here.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "spark_attn.h"

namespace spark {

// u_k = theta^(-2k/r) / (2 pi) as an unevaluated fp32 pair (hi, lo).
void fill_rope_table(const spark_layer_desc *d, RopeTable *t) {
    std::memset(t, 0, sizeof(*t));
    t->rot_dim = d->rot_dim;
    const double two_pi = 6.283185307179586476925286766559;
    for (int k = 0; k < d->rot_dim / 2; ++k) {
        const double inv_freq = std::pow(d->rope_theta, -2.0 * k / d->rot_dim);
        const double u = inv_freq / two_pi;
        const float hi = static_cast<float>(u);
        const float lo = static_cast<float>(u - static_cast<double>(hi));
        t->u[k] = make_float2(hi, lo);
    }
}

cudaError_t launch_decode(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const DecodeParams &P,
                          cudaStream_t stream);
cudaError_t launch_prefill(const CUtensorMap &tm_q, const CUtensorMap &tm_kv_k,
                           const CUtensorMap &tm_kv_v, const CUtensorMap &tm_krot,
                           const CUtensorMap &tm_out, const PrefillParams &P, cudaStream_t stream);

namespace {

constexpr int kFallbackSms = 152;  // GB300 SM count, used when no device is visible

// ------------------------------------------------------------ device facts

struct DeviceInfo {
    std::atomic<int> ready{0};
    int sms = 0;
    int major = 0, minor = 0;
};
DeviceInfo g_devices[64];
std::mutex g_device_mutex;

// SM count and compute capability of the current device (cached per device).
// Returns false when no device is usable.
bool current_device(int *sms, int *major, int *minor) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return false;
    }
    DeviceInfo &d = g_devices[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_device_mutex);
        if (!d.ready.load(std::memory_order_relaxed)) {
            if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) !=
                    cudaSuccess ||
                cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) !=
                    cudaSuccess) {
                cudaGetLastError();
                return false;
            }
            d.ready.store(1, std::memory_order_release);
        }
    }
    *sms = d.sms;
    *major = d.major;
    *minor = d.minor;
    return true;
}

int sm_count_or_default() {
    int sms, major, minor;
    if (current_device(&sms, &major, &minor)) return sms;
    return kFallbackSms;
}

// The kernels are built for sm_103a only.
spark_status check_device() {
    int sms, major, minor;
    if (!current_device(&sms, &major, &minor)) return SPARK_ERR_CUDA;
    if (major != 10 || minor != 3) return SPARK_ERR_DEVICE;
    return SPARK_OK;
}

// ------------------------------------------------------------ tensor maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        cudaGetLastError();
    });
    return fn;
}

// bf16 tiled map: dims innermost first, strides in bytes for dims 1..rank-1.
bool encode_bf16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                 const uint64_t *strides, const uint32_t *box, CUtensorMapSwizzle swizzle) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) gs[i] = strides[i];
    }
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), gd, gs,
                    bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------ validation

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

spark_status check_layer(const spark_layer_desc *d, int H, int Hkv) {
    if (!d) return SPARK_ERR_NULL;
    if (H < 0 || Hkv < 0) return SPARK_ERR_SHAPE;
    if (H == 0 || Hkv == 0 || H % Hkv != 0) return SPARK_ERR_SHAPE;
    if (d->kind != SPARK_LAYER_FULL && d->kind != SPARK_LAYER_SLIDING) return SPARK_ERR_SHAPE;
    if (d->kind == SPARK_LAYER_SLIDING && d->window < 1) return SPARK_ERR_SHAPE;
    if (!(d->rope_theta > 0.0) || !std::isfinite(d->rope_theta)) return SPARK_ERR_SHAPE;
    if (d->rot_dim < 0 || d->rot_dim > SPARK_HEAD_DIM || (d->rot_dim & 1)) return SPARK_ERR_SHAPE;
    if (d->rot_dim % 16 != 0) return SPARK_ERR_UNSUPPORTED;
    if (d->gate_mode != SPARK_GATE_SIGMOID && d->gate_mode != SPARK_GATE_SILU)
        return SPARK_ERR_UNSUPPORTED;
    const int G = H / Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8) return SPARK_ERR_UNSUPPORTED;
    return SPARK_OK;
}

spark_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return SPARK_OK;
    cudaGetLastError();
    return SPARK_ERR_CUDA;
}

// ------------------------------------------------------------ decode plan

struct DecodePlan {
    int nsplit;
    int chunk;
    size_t ml_offset, o_offset, bytes;
};

// Splits the scanned slots of each (sequence, KV head) into equal chunks of a
// multiple of 64 slots.  When there are fewer (sequence, KV head) pairs than
// SMs, the chunks fill exactly one wave of the GPU (one CTA per SM streams one
// long chunk, so no CTA starts late and few partial states are left to
// merge); otherwise chunks of at most 4096 slots keep ragged batches balanced.
DecodePlan plan_decode(int B, int H, int Hkv, int64_t cap, const spark_layer_desc *d, int sms) {
    DecodePlan pl{};
    long long max_scan = (d->kind == SPARK_LAYER_FULL) ? cap - 1 : cap;
    if (max_scan < 1) max_scan = 1;
    const long long kMaxChunk = 4096;
    const long long units = static_cast<long long>(B) * Hkv;
    long long ns = (max_scan + kMaxChunk - 1) / kMaxChunk;
    if (units > 0 && units <= sms) ns = sms / units;
    const long long max_ns = (max_scan + 63) / 64;
    if (ns > max_ns) ns = max_ns;
    if (ns < 1) ns = 1;
    long long chunk = (max_scan + ns - 1) / ns;
    chunk = (chunk + 63) / 64 * 64;
    ns = (max_scan + chunk - 1) / chunk;
    pl.nsplit = static_cast<int>(ns);
    pl.chunk = static_cast<int>(chunk);
    const size_t parts = static_cast<size_t>(B) * H * pl.nsplit;
    pl.ml_offset = kWorkspaceHeader;
    pl.o_offset = align_up(pl.ml_offset + parts * 2 * sizeof(float), 256);
    pl.bytes = align_up(pl.o_offset + parts * kHeadDim * sizeof(float), 256);
    return pl;
}

spark_status check_decode(int B, int H, int Hkv, int64_t cap, const spark_layer_desc *d) {
    spark_status st = check_layer(d, H, Hkv);
    if (st != SPARK_OK) return st;
    if (B < 0) return SPARK_ERR_SHAPE;
    if (cap < 1) return SPARK_ERR_CAPACITY;
    if (d->kind == SPARK_LAYER_SLIDING && cap < d->window) return SPARK_ERR_CAPACITY;
    if (cap > 0x7fffffffLL) return SPARK_ERR_UNSUPPORTED;
    return SPARK_OK;
}

// ------------------------------------------------------------ prefill plan

constexpr int kPrefillRows = 128;  // query rows (token x head) per CTA tile

struct PrefillPlan {
    int rot_w;          // leading K dims stored rotated (rot_dim rounded up to 64)
    size_t krot_offset, bytes;
};

PrefillPlan plan_prefill(int B, int T, int Hkv, const spark_layer_desc *d) {
    PrefillPlan pl{};
    pl.rot_w = (d->rot_dim + 63) / 64 * 64;
    pl.krot_offset = kWorkspaceHeader;
    pl.bytes = align_up(pl.krot_offset + static_cast<size_t>(B) * Hkv * T * pl.rot_w * 2, 256);
    return pl;
}

spark_status check_prefill(int B, int T, int H, int Hkv, const spark_layer_desc *d) {
    spark_status st = check_layer(d, H, Hkv);
    if (st != SPARK_OK) return st;
    if (B < 0 || T < 0) return SPARK_ERR_SHAPE;
    if (static_cast<long long>(B) * T > 0x7fffffffLL) return SPARK_ERR_UNSUPPORTED;
    return SPARK_OK;
}

}  // namespace

// Prefill, optionally filling the decode cache (k_cache != nullptr), or a
// chunked prefill over a cache that already holds start[b] tokens.  With
// validate_only, returns after the host-side checks and enqueues nothing.
spark_status prefill_impl(const void *qkv, const float *gate, const int32_t *pos,
                          const spark_layer_desc *desc, int B, int T, int H, int Hkv, void *out,
                          void *k_cache, void *v_cache, int64_t cap, const int32_t *start,
                          void *workspace, size_t workspace_bytes, void *stream,
                          bool validate_only) {
    spark_status st = check_prefill(B, T, H, Hkv, desc);
    if (st != SPARK_OK) return st;
    if (k_cache || v_cache) {
        if (cap < 1) return SPARK_ERR_CAPACITY;
        if (desc->kind == SPARK_LAYER_FULL && cap < T) return SPARK_ERR_CAPACITY;
        if (desc->kind == SPARK_LAYER_SLIDING && cap < desc->window) return SPARK_ERR_CAPACITY;
        if (cap > 0x7fffffffLL) return SPARK_ERR_UNSUPPORTED;
        if (start && desc->kind == SPARK_LAYER_SLIDING) {
            // the chunk's writes must not overwrite keys its own rows still see
            if (cap < static_cast<int64_t>(desc->window) + T - 1) return SPARK_ERR_CAPACITY;
            if (cap % 128 != 0) return SPARK_ERR_UNSUPPORTED;
        }
    }
    if (B == 0 || T == 0) return SPARK_OK;
    if (!qkv || !gate || !pos || !out || !workspace) return SPARK_ERR_NULL;
    if ((k_cache == nullptr) != (v_cache == nullptr)) return SPARK_ERR_NULL;
    if (!aligned(qkv, 16) || !aligned(out, 16) || !aligned(gate, 4) || !aligned(pos, 4) ||
        !aligned(workspace, 256) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(start, 4))
        return SPARK_ERR_ALIGN;
    const PrefillPlan pl = plan_prefill(B, T, Hkv, desc);
    if (workspace_bytes < pl.bytes) return SPARK_ERR_WORKSPACE;
    st = check_device();
    if (st != SPARK_OK || validate_only) return st;

    const int G = H / Hkv;
    const int tq = kPrefillRows / G;  // tokens per query tile
    PrefillParams P;
    std::memset(&P, 0, sizeof(P));
    P.qkv = static_cast<const __nv_bfloat16 *>(qkv);
    P.gate = gate;
    P.pos = pos;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    P.status = reinterpret_cast<unsigned *>(ws);
    P.krot = reinterpret_cast<__nv_bfloat16 *>(ws + pl.krot_offset);
    P.k_cache = static_cast<__nv_bfloat16 *>(k_cache);
    P.v_cache = static_cast<__nv_bfloat16 *>(v_cache);
    P.cap = k_cache ? cap : 0;
    P.start = start;
    P.B = B;
    P.T = T;
    P.H = H;
    P.Hkv = Hkv;
    P.G = G;
    P.kind = desc->kind;
    P.window = desc->kind == SPARK_LAYER_SLIDING ? desc->window : 0;
    P.gate_mode = desc->gate_mode;
    P.rot_w = pl.rot_w;
    P.n_qtiles = (T + tq - 1) / tq;
    P.wave = sm_count_or_default();
    fill_rope_table(desc, &P.rope);

    const uint64_t heads = static_cast<uint64_t>(H + 2 * Hkv);
    CUtensorMap tm_q, tm_kv_k, tm_kv_v, tm_krot, tm_out;
    std::memset(&tm_krot, 0, sizeof(tm_krot));
    {
        // qkv as [B][T][heads][256]
        const uint64_t dims[4] = {kHeadDim, heads, static_cast<uint64_t>(T),
                                  static_cast<uint64_t>(B)};
        const uint64_t strides[3] = {kHeadDim * 2ull, heads * kHeadDim * 2ull,
                                     static_cast<uint64_t>(T) * heads * kHeadDim * 2ull};
        const uint32_t box_q[4] = {64, static_cast<uint32_t>(G), static_cast<uint32_t>(tq), 1};
        const uint32_t box_k[4] = {64, 1, 128, 1};
        const uint32_t box_v[4] = {64, 1, 32, 1};
        if (!encode_bf16(&tm_q, qkv, 4, dims, strides, box_q, CU_TENSOR_MAP_SWIZZLE_128B))
            return SPARK_ERR_CUDA;
        if (start) {
            // chunked prefill: keys and values come from the caches [B][Hkv][cap][256]
            const uint64_t cdims[4] = {kHeadDim, static_cast<uint64_t>(cap),
                                       static_cast<uint64_t>(Hkv), static_cast<uint64_t>(B)};
            const uint64_t cstrides[3] = {kHeadDim * 2ull,
                                          static_cast<uint64_t>(cap) * kHeadDim * 2ull,
                                          static_cast<uint64_t>(Hkv) * cap * kHeadDim * 2ull};
            const uint32_t cbox_k[4] = {64, 128, 1, 1};
            const uint32_t cbox_v[4] = {64, 32, 1, 1};
            if (!encode_bf16(&tm_kv_k, k_cache, 4, cdims, cstrides, cbox_k,
                             CU_TENSOR_MAP_SWIZZLE_128B) ||
                !encode_bf16(&tm_kv_v, v_cache, 4, cdims, cstrides, cbox_v,
                             CU_TENSOR_MAP_SWIZZLE_128B))
                return SPARK_ERR_CUDA;
        } else if (!encode_bf16(&tm_kv_k, qkv, 4, dims, strides, box_k,
                                CU_TENSOR_MAP_SWIZZLE_128B) ||
                   !encode_bf16(&tm_kv_v, qkv, 4, dims, strides, box_v,
                                CU_TENSOR_MAP_SWIZZLE_128B)) {
            return SPARK_ERR_CUDA;
        }
    }
    if (pl.rot_w > 0) {
        // rotated K as [B*Hkv][T][rot_w]
        const uint64_t dims[3] = {static_cast<uint64_t>(pl.rot_w), static_cast<uint64_t>(T),
                                  static_cast<uint64_t>(B) * Hkv};
        const uint64_t strides[2] = {pl.rot_w * 2ull,
                                     static_cast<uint64_t>(T) * pl.rot_w * 2ull};
        const uint32_t box[3] = {64, 128, 1};
        if (!encode_bf16(&tm_krot, P.krot, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return SPARK_ERR_CUDA;
    }
    {
        // out as [B][T][H][256]
        const uint64_t dims[4] = {kHeadDim, static_cast<uint64_t>(H), static_cast<uint64_t>(T),
                                  static_cast<uint64_t>(B)};
        const uint64_t strides[3] = {kHeadDim * 2ull, static_cast<uint64_t>(H) * kHeadDim * 2ull,
                                     static_cast<uint64_t>(T) * H * kHeadDim * 2ull};
        const uint32_t box[4] = {64, static_cast<uint32_t>(G), static_cast<uint32_t>(tq), 1};
        if (!encode_bf16(&tm_out, out, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return SPARK_ERR_CUDA;
    }
    return from_cuda(launch_prefill(tm_q, tm_kv_k, tm_kv_v, tm_krot, tm_out, P,
                                    static_cast<cudaStream_t>(stream)));
}

// One decode step; with validate_only, returns after the host-side checks.
spark_status decode_impl(const void *qkv, const float *gate, const int32_t *pos, void *k_cache,
                         void *v_cache, int64_t cap, const spark_layer_desc *desc, int B, int H,
                         int Hkv, void *out, void *workspace, size_t workspace_bytes,
                         void *stream, bool validate_only) {
    spark_status st = check_decode(B, H, Hkv, cap, desc);
    if (st != SPARK_OK) return st;
    if (B == 0) return SPARK_OK;
    if (!qkv || !gate || !pos || !k_cache || !v_cache || !out || !workspace) return SPARK_ERR_NULL;
    if (!aligned(qkv, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(gate, 4) || !aligned(pos, 4) || !aligned(workspace, 256))
        return SPARK_ERR_ALIGN;
    const DecodePlan pl = plan_decode(B, H, Hkv, cap, desc, sm_count_or_default());
    if (workspace_bytes < pl.bytes) return SPARK_ERR_WORKSPACE;
    st = check_device();
    if (st != SPARK_OK || validate_only) return st;

    DecodeParams P;
    std::memset(&P, 0, sizeof(P));
    P.qkv = static_cast<const __nv_bfloat16 *>(qkv);
    P.gate = gate;
    P.pos = pos;
    P.k_cache = static_cast<__nv_bfloat16 *>(k_cache);
    P.v_cache = static_cast<__nv_bfloat16 *>(v_cache);
    P.out = static_cast<__nv_bfloat16 *>(out);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    P.status = reinterpret_cast<unsigned *>(ws);
    P.part_ml = reinterpret_cast<float *>(ws + pl.ml_offset);
    P.part_o = reinterpret_cast<float *>(ws + pl.o_offset);
    P.cap = cap;
    P.B = B;
    P.H = H;
    P.Hkv = Hkv;
    P.G = H / Hkv;
    P.kind = desc->kind;
    P.window = desc->kind == SPARK_LAYER_SLIDING ? desc->window : 0;
    P.gate_mode = desc->gate_mode;
    P.nsplit = pl.nsplit;
    P.chunk = pl.chunk;
    P.counters = reinterpret_cast<unsigned *>(ws) + 1;  // header words after the status word
    P.fuse_merge = decode_fuses_merge(pl.nsplit, static_cast<long long>(B) * Hkv, true) ? 1 : 0;
    fill_rope_table(desc, &P.rope);

    // caches as [B][Hkv][cap][256]; boxes of 64 slots x 64 dims (128-byte rows)
    CUtensorMap tm_k, tm_v;
    const uint64_t dims[4] = {static_cast<uint64_t>(kHeadDim), static_cast<uint64_t>(cap),
                              static_cast<uint64_t>(Hkv), static_cast<uint64_t>(B)};
    const uint64_t strides[3] = {kHeadDim * 2ull, static_cast<uint64_t>(cap) * kHeadDim * 2ull,
                                 static_cast<uint64_t>(Hkv) * cap * kHeadDim * 2ull};
    const uint32_t box[4] = {64, 64, 1, 1};
    if (!encode_bf16(&tm_k, k_cache, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_bf16(&tm_v, v_cache, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return SPARK_ERR_CUDA;
    return from_cuda(launch_decode(tm_k, tm_v, P, static_cast<cudaStream_t>(stream)));
}

}  // namespace spark

using namespace spark;

extern "C" {

const char *spark_status_str(spark_status s) {
    switch (s) {
        case SPARK_OK: return "ok";
        case SPARK_ERR_NULL: return "a required pointer is NULL";
        case SPARK_ERR_SHAPE: return "a size is negative or inconsistent";
        case SPARK_ERR_UNSUPPORTED: return "valid arguments that the library does not support";
        case SPARK_ERR_ALIGN: return "a pointer is not aligned (16 bytes; workspace 256 bytes)";
        case SPARK_ERR_CAPACITY: return "the KV cache is too small for the layer";
        case SPARK_ERR_WORKSPACE: return "workspace missing or too small";
        case SPARK_ERR_CUDA: return "a CUDA call failed while enqueuing work";
        case SPARK_ERR_DEVICE: return "the current device is not an sm_103 GPU";
    }
    return "unknown status";
}

const char *spark_attn_version(void) { return "0.1.0"; }

size_t spark_attn_decode_workspace_size(int B, int H, int Hkv, int64_t cap,
                                        const spark_layer_desc *desc) {
    if (check_decode(B, H, Hkv, cap, desc) != SPARK_OK) return 0;
    return plan_decode(B, H, Hkv, cap, desc, sm_count_or_default()).bytes;
}

int spark_attn_decode_launch_count(int B, int H, int Hkv, int64_t cap,
                                   const spark_layer_desc *desc) {
    if (check_decode(B, H, Hkv, cap, desc) != SPARK_OK || B == 0) return 0;
    const DecodePlan pl = plan_decode(B, H, Hkv, cap, desc, sm_count_or_default());
    return decode_fuses_merge(pl.nsplit, static_cast<long long>(B) * Hkv, true) ? 1 : 2;
}

spark_status spark_attn_decode(const void *qkv, const float *gate, const int32_t *pos,
                               void *k_cache, void *v_cache, int64_t cap,
                               const spark_layer_desc *desc, int B, int H, int Hkv, void *out,
                               void *workspace, size_t workspace_bytes, void *stream) {
    return decode_impl(qkv, gate, pos, k_cache, v_cache, cap, desc, B, H, Hkv, out, workspace,
                       workspace_bytes, stream, false);
}

size_t spark_attn_prefill_workspace_size(int B, int T, int H, int Hkv,
                                         const spark_layer_desc *desc) {
    if (check_prefill(B, T, H, Hkv, desc) != SPARK_OK) return 0;
    return plan_prefill(B, T, Hkv, desc).bytes;
}

extern "C" spark_status spark_attn_prefill(const void *qkv, const float *gate, const int32_t *pos,
                                           const spark_layer_desc *desc, int B, int T, int H,
                                           int Hkv, void *out, void *workspace,
                                           size_t workspace_bytes, void *stream) {
    return prefill_impl(qkv, gate, pos, desc, B, T, H, Hkv, out, nullptr, nullptr, 0, nullptr,
                        workspace, workspace_bytes, stream, false);
}

extern "C" spark_status spark_attn_prefill_cache(const void *qkv, const float *gate,
                                                 const int32_t *pos, void *k_cache,
                                                 void *v_cache, int64_t cap,
                                                 const spark_layer_desc *desc, int B, int T,
                                                 int H, int Hkv, void *out, void *workspace,
                                                 size_t workspace_bytes, void *stream) {
    const spark_status st = check_prefill(B, T, H, Hkv, desc);
    if (st != SPARK_OK) return st;
    if (B == 0 || T == 0) return SPARK_OK;
    if (!k_cache || !v_cache) return SPARK_ERR_NULL;
    return prefill_impl(qkv, gate, pos, desc, B, T, H, Hkv, out, k_cache, v_cache, cap, nullptr,
                        workspace, workspace_bytes, stream, false);
}

extern "C" spark_status spark_attn_prefill_chunk(const void *qkv, const float *gate,
                                                 const int32_t *pos, void *k_cache,
                                                 void *v_cache, int64_t cap,
                                                 const int32_t *start,
                                                 const spark_layer_desc *desc, int B, int T,
                                                 int H, int Hkv, void *out, void *workspace,
                                                 size_t workspace_bytes, void *stream) {
    const spark_status st = check_prefill(B, T, H, Hkv, desc);
    if (st != SPARK_OK) return st;
    if (B == 0 || T == 0) return SPARK_OK;
    if (!k_cache || !v_cache || !start) return SPARK_ERR_NULL;
    return prefill_impl(qkv, gate, pos, desc, B, T, H, Hkv, out, k_cache, v_cache, cap, start,
                        workspace, workspace_bytes, stream, false);
}

spark_status spark_attn_read_status(void *workspace, uint32_t *status_out, int clear,
                                    void *stream) {
    if (!workspace || !status_out) return SPARK_ERR_NULL;
    if (!aligned(workspace, 256)) return SPARK_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t value = 0;
    if (cudaMemcpyAsync(&value, workspace, sizeof(value), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return SPARK_ERR_CUDA;
    }
    if (clear) {
        if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess) {
            cudaGetLastError();
            return SPARK_ERR_CUDA;
        }
    }
    *status_out = value;
    return SPARK_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- no-alloc decode
//
// A decode entry point for callers that cannot hand the library a workspace:
// code running under a memory manager that owns every byte of device memory
// (a serving runtime that reserves its pool up front, a plugin host that
// passes only inputs and outputs), or code on a path where cudaMalloc is off
// limits because it synchronizes the device.  The split-KV partial states
// that spark_attn_decode keeps in the caller's workspace live here in one
// fixed buffer owned by the library instead.  Every device that loads the
// library holds this buffer until the process exits.

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // SPARK_NOALLOC_SCRATCH_BYTES

// In host code this name is only a stand-in for the device buffer: the
// device address comes from cudaGetSymbolAddress (see noalloc_scratch).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;

// The buffer's device address per device, with the context it was looked up
// in: a device reset rebuilds the primary context and reloads the module, so
// an address is reused only while the same context is current.
struct NoAllocAddr {
    CUcontext ctx = nullptr;
    void *ptr = nullptr;
};
NoAllocAddr g_noalloc_addr[64];

using CtxGetCurrentFn = CUresult (*)(CUcontext *);

CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
        cudaGetLastError();
    });
    return fn;
}

CUcontext current_context() {
    CtxGetCurrentFn fn = ctx_get_current_fn();
    CUcontext ctx = nullptr;
    if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
    return ctx;
}

// Device address of the scratch buffer on the current device, looked up with
// that device current: once per device, and again whenever another context is
// current than the one of the last lookup.  Returns nullptr on failure.
void *noalloc_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoAllocAddr &a = g_noalloc_addr[dev];
    if (a.ptr && a.ctx != nullptr && a.ctx == current_context()) return a.ptr;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
        cudaGetLastError();
        a = NoAllocAddr();
        return nullptr;
    }
    // the lookup made the device's context current if it was not yet
    a.ctx = current_context();
    a.ptr = p;
    return p;
}

}  // namespace

extern "C" spark_status spark_attn_decode_noalloc(const void *qkv, const float *gate,
                                                  const int32_t *pos, void *k_cache,
                                                  void *v_cache, int64_t cap,
                                                  const spark_layer_desc *desc, int B, int H,
                                                  int Hkv, void *out, uint32_t *device_status,
                                                  void *stream) {
    spark_status st = check_decode(B, H, Hkv, cap, desc);
    if (st != SPARK_OK) return st;
    if (B == 0) return SPARK_OK;
    if (!qkv || !gate || !pos || !k_cache || !v_cache || !out) return SPARK_ERR_NULL;
    if (!aligned(qkv, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(gate, 4) || !aligned(pos, 4) || (device_status && !aligned(device_status, 4)))
        return SPARK_ERR_ALIGN;
    const DecodePlan pl = plan_decode(B, H, Hkv, cap, desc, sm_count_or_default());
    if (pl.bytes > kNoAllocScratchBytes) return SPARK_ERR_WORKSPACE;
    st = check_device();
    if (st != SPARK_OK) return st;
    uint8_t *ws = static_cast<uint8_t *>(noalloc_scratch());
    if (!ws) return SPARK_ERR_CUDA;

    DecodeParams P;
    std::memset(&P, 0, sizeof(P));
    P.qkv = static_cast<const __nv_bfloat16 *>(qkv);
    P.gate = gate;
    P.pos = pos;
    P.k_cache = static_cast<__nv_bfloat16 *>(k_cache);
    P.v_cache = static_cast<__nv_bfloat16 *>(v_cache);
    P.out = static_cast<__nv_bfloat16 *>(out);
    // Device-side fault bits go to the caller's word when one is given, else
    // to a word of the scratch buffer that nobody reads.
    P.status = device_status ? reinterpret_cast<unsigned *>(device_status)
                             : reinterpret_cast<unsigned *>(ws);
    P.part_ml = reinterpret_cast<float *>(ws + pl.ml_offset);
    P.part_o = reinterpret_cast<float *>(ws + pl.o_offset);
    P.cap = cap;
    P.B = B;
    P.H = H;
    P.Hkv = Hkv;
    P.G = H / Hkv;
    P.kind = desc->kind;
    P.window = desc->kind == SPARK_LAYER_SLIDING ? desc->window : 0;
    P.gate_mode = desc->gate_mode;
    P.nsplit = pl.nsplit;
    P.chunk = pl.chunk;
    // the scratch buffer is never zeroed, so it holds no split counters: the
    // split kernel merges only where it is the only split
    P.counters = nullptr;
    P.fuse_merge = decode_fuses_merge(pl.nsplit, static_cast<long long>(B) * Hkv, false) ? 1 : 0;
    fill_rope_table(desc, &P.rope);

    CUtensorMap tm_k, tm_v;
    const uint64_t dims[4] = {static_cast<uint64_t>(kHeadDim), static_cast<uint64_t>(cap),
                              static_cast<uint64_t>(Hkv), static_cast<uint64_t>(B)};
    const uint64_t strides[3] = {kHeadDim * 2ull, static_cast<uint64_t>(cap) * kHeadDim * 2ull,
                                 static_cast<uint64_t>(Hkv) * cap * kHeadDim * 2ull};
    const uint32_t box[4] = {64, 64, 1, 1};
    if (!encode_bf16(&tm_k, k_cache, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_bf16(&tm_v, v_cache, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return SPARK_ERR_CUDA;
    return from_cuda(launch_decode(tm_k, tm_v, P, static_cast<cudaStream_t>(stream)));
}
