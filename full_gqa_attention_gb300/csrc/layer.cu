// layer.cu -- the attention block around the core: q_k_v_proj and g_proj on
// the normed hidden state, the core (prefill or one decode step), out_proj.
//
// Spark-X2.5 architecture (4B / 1.7B), §3 Eq. 1 and Fig. 1: a fused
// q_k_v_proj (hidden -> (H + 2 Hkv) * 256) and a separate g_proj (hidden -> H,
// one gate logit per head) read the normed hidden state; out_proj
// (H * 256 -> hidden) maps the gated attention output back.  §1: the
// checkpoints run in bfloat16 and the pages list no biases.
//
// With more than a few rows the projections run on the tcgen05 GEMM of
// gemm.cu (bf16 operands, fp32 accumulation in TMEM): q_k_v_proj and g_proj
// in one launch, whose g_proj columns leave the kernel as fp32 values rounded
// to bf16, the dtype of the Linear's output, before the core's epilogue takes
// the gate activation of them in fp32; then out_proj.  In a prefill the same
// epilogue also rotates Q and K (RoPE of §4, from the bf16-rounded products,
// as the core would), so the core runs without its rotation kernel and
// without rotating Q in the attention kernel.  With at most kGemvMaxM
// rows (a decode step) they are weight-streaming GEMVs of this file, g_proj
// in the same pass as q_k_v_proj.
#include "common.cuh"
#include "spark_attn.h"

namespace spark {

spark_status launch_linear(const void *x, const void *w, void *y, long long M, int N, int K,
                           const void *w2, float *y2, int N2, unsigned *status,
                           cudaStream_t stream, const RopeTable *rope, const int32_t *pos,
                           int rope_heads);
void fill_rope_table(const spark_layer_desc *d, RopeTable *t);
spark_status check_linear(const void *x, const void *w, void *y, long long M, int N, int K,
                          const void *w2, float *y2, int N2);
spark_status prefill_impl(const void *qkv, const float *gate, const int32_t *pos,
                          const spark_layer_desc *desc, int B, int T, int H, int Hkv, void *out,
                          void *k_cache, void *v_cache, int64_t cap, const int32_t *start,
                          void *workspace, size_t workspace_bytes, void *stream,
                          bool validate_only);
spark_status decode_impl(const void *qkv, const float *gate, const int32_t *pos, void *k_cache,
                         void *v_cache, int64_t cap, const spark_layer_desc *desc, int B, int H,
                         int Hkv, void *out, void *workspace, size_t workspace_bytes,
                         void *stream, bool validate_only);

namespace {

// ---------------------------------------------------------------- decode GEMV
//
// A decode step projects one hidden state per sequence: y = W x for a few
// vectors x, which reads the whole weight matrix once and is bound by that
// read.  Each warp takes one weight row and streams it in blocks of
// kGemvBlk coalesced 16-byte loads per lane, all issued before any of them is
// used (the few x vectors come from L1), accumulates in fp32, reduces over
// the warp and rounds once to bf16.  One launch can cover two matrices (the
// rows of W_qkv, then those of W_g), so g_proj rides along with q_k_v_proj.

constexpr int kGemvWarps = 8;     // warps (rows) per CTA
constexpr int kGemvBlk = 8;       // 16-byte loads in flight per lane
constexpr int kGemvMaxM = 8;      // vectors per launch

struct GemvSeg {
    const __nv_bfloat16 *w;       // [n][K] row-major
    void *out;                    // [M][n]: bf16, or fp32 holding bf16-rounded values
    int n;                        // rows
    int out_f32;                  // output type
};

__global__ void __launch_bounds__(kGemvWarps * 32) gemv_kernel(GemvSeg s0, GemvSeg s1,
                                                               const __nv_bfloat16 *x, int M,
                                                               int K) {
    grid_dep_wait();  // x may come from the previous kernel
    grid_dep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = blockIdx.x * kGemvWarps + warp;
    if (n >= s0.n + s1.n) return;
    const bool first = n < s0.n;
    const GemvSeg &sg = first ? s0 : s1;
    const int nn = first ? n : n - s0.n;
    const __nv_bfloat16 *w = sg.w + static_cast<size_t>(nn) * K;
    float acc[kGemvMaxM];
#pragma unroll
    for (int m = 0; m < kGemvMaxM; ++m) acc[m] = 0.f;
    for (int kb = 0; kb < K; kb += 32 * 8 * kGemvBlk) {
        uint4 wv[kGemvBlk];
#pragma unroll
        for (int c = 0; c < kGemvBlk; ++c) {
            const int k = kb + (c * 32 + lane) * 8;
            wv[c] = (k < K) ? __ldcs(reinterpret_cast<const uint4 *>(w + k)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int c = 0; c < kGemvBlk; ++c) {
            const int k = kb + (c * 32 + lane) * 8;
            if (k >= K) break;
            const uint32_t ww[4] = {wv[c].x, wv[c].y, wv[c].z, wv[c].w};
#pragma unroll
            for (int m = 0; m < kGemvMaxM; ++m) {
                if (m >= M) break;
                const uint4 xv =
                    __ldg(reinterpret_cast<const uint4 *>(x + static_cast<size_t>(m) * K + k));
                const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[m] = fmaf(bf16_lo(ww[i]), bf16_lo(xw[i]), acc[m]);
                    acc[m] = fmaf(bf16_hi(ww[i]), bf16_hi(xw[i]), acc[m]);
                }
            }
        }
    }
#pragma unroll
    for (int m = 0; m < kGemvMaxM; ++m) {
        if (m >= M) break;
        float v = acc[m];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) {
            const __nv_bfloat16 b = __float2bfloat16_rn(v);
            if (sg.out_f32)
                static_cast<float *>(sg.out)[static_cast<size_t>(m) * sg.n + nn] = __bfloat162float(b);
            else
                static_cast<__nv_bfloat16 *>(sg.out)[static_cast<size_t>(m) * sg.n + nn] = b;
        }
    }
}

cudaError_t launch_gemv(const GemvSeg &s0, const GemvSeg &s1, const void *x, int M, int K,
                        cudaStream_t stream) {
    const long long rows = static_cast<long long>(s0.n) + s1.n;
    const unsigned grid = static_cast<unsigned>((rows + kGemvWarps - 1) / kGemvWarps);
    return launch_overlapped(gemv_kernel, dim3(grid), dim3(kGemvWarps * 32), 0, stream, s0, s1,
                             static_cast<const __nv_bfloat16 *>(x), M, K);
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// The layer workspace: the core's workspace first (its status word is the
// layer's), then qkv, gate logits and the gated attention output.
struct LayerPlan {
    size_t core, qkv, gate, attn, bytes;
};

LayerPlan plan_layer(size_t core_bytes, long long rows, int H, int Hkv) {
    LayerPlan pl{};
    pl.core = 0;
    pl.qkv = align256(core_bytes);
    pl.gate = pl.qkv + align256(static_cast<size_t>(rows) * (H + 2 * Hkv) * kHeadDim * 2);
    pl.attn = pl.gate + align256(static_cast<size_t>(rows) * H * 4);
    pl.bytes = pl.attn + align256(static_cast<size_t>(rows) * H * kHeadDim * 2);
    return pl;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The GEMM's own checks of both projections, before anything is enqueued
// (rows above the GEMV's limit only: the GEMV has none to fail).
spark_status check_layer_linears(const void *x, const void *w_qkv, const void *w_g,
                                 const void *w_o, void *y, long long rows, int hidden, int H,
                                 int Hkv, uint8_t *ws, const LayerPlan &pl) {
    if (rows <= kGemvMaxM) return SPARK_OK;
    spark_status st = check_linear(x, w_qkv, ws + pl.qkv, rows, (H + 2 * Hkv) * kHeadDim, hidden,
                                   w_g, reinterpret_cast<float *>(ws + pl.gate), H);
    if (st != SPARK_OK) return st;
    return check_linear(ws + pl.attn, w_o, y, rows, hidden, H * kHeadDim, nullptr, nullptr, 0);
}

spark_status check_hidden(int hidden) {
    if (hidden <= 0) return SPARK_ERR_SHAPE;
    if (hidden % 8 != 0) return SPARK_ERR_UNSUPPORTED;  // rows of 16 bytes
    return SPARK_OK;
}

// Whether a prefill block rotates Q and K in the q_k_v_proj epilogue (the GEMM
// path, and rotated widths it handles: r/2 a multiple of 32, so 64 and 256,
// the two Spark-X2.5 layer types); the core then runs without rotating.
bool rope_in_projection(long long rows, const spark_layer_desc *d) {
    return rows > kGemvMaxM && d->rot_dim > 0 && (d->rot_dim / 2) % 32 == 0;
}

// q_k_v_proj and g_proj of `rows` hidden states into the workspace; with
// `rope`, Q and K leave the GEMM rotated at the positions `pos`.
spark_status project_in(const void *x, const void *w_qkv, const void *w_g, long long rows,
                        int hidden, int H, int Hkv, uint8_t *ws, const LayerPlan &pl,
                        cudaStream_t stream, const RopeTable *rope = nullptr,
                        const int32_t *pos = nullptr) {
    const int M = static_cast<int>(rows);
    if (M <= kGemvMaxM) {
        // a few hidden states: one weight-streaming pass over W_qkv and W_g
        const GemvSeg qkv{static_cast<const __nv_bfloat16 *>(w_qkv), ws + pl.qkv,
                          (H + 2 * Hkv) * kHeadDim, 0};
        const GemvSeg gate{static_cast<const __nv_bfloat16 *>(w_g), ws + pl.gate, H, 1};
        return launch_gemv(qkv, gate, x, M, hidden, stream) == cudaSuccess ? SPARK_OK
                                                                           : SPARK_ERR_CUDA;
    }
    // both products in one launch; the status word is the core's (workspace start)
    return launch_linear(x, w_qkv, ws + pl.qkv, rows, (H + 2 * Hkv) * kHeadDim, hidden, w_g,
                         reinterpret_cast<float *>(ws + pl.gate), H,
                         reinterpret_cast<unsigned *>(ws), stream, rope, pos,
                         rope ? H + Hkv : 0);
}

// out_proj of `rows` gated attention outputs: y = a W_o^T.
spark_status project_out(const void *attn, const void *w_o, void *y, long long rows, int hidden,
                         int H, uint8_t *ws, cudaStream_t stream) {
    const int M = static_cast<int>(rows);
    if (M <= kGemvMaxM) {
        const GemvSeg out{static_cast<const __nv_bfloat16 *>(w_o), y, hidden, 0};
        const GemvSeg none{nullptr, nullptr, 0, 0};
        return launch_gemv(out, none, attn, M, H * kHeadDim, stream) == cudaSuccess
                   ? SPARK_OK
                   : SPARK_ERR_CUDA;
    }
    return launch_linear(attn, w_o, y, rows, hidden, H * kHeadDim, nullptr, nullptr, 0,
                         reinterpret_cast<unsigned *>(ws), stream, nullptr, nullptr, 0);
}

}  // namespace
}  // namespace spark

using namespace spark;

extern "C" {

size_t spark_attn_layer_prefill_workspace_size(int B, int T, int hidden, int H, int Hkv,
                                               const spark_layer_desc *desc) {
    if (check_hidden(hidden) != SPARK_OK) return 0;
    const size_t core = spark_attn_prefill_workspace_size(B, T, H, Hkv, desc);
    if (core == 0) return 0;
    return plan_layer(core, static_cast<long long>(B) * T, H, Hkv).bytes;
}

spark_status spark_attn_layer_prefill(const void *x, const void *w_qkv, const void *w_g,
                                      const void *w_o, const int32_t *pos, void *k_cache,
                                      void *v_cache, int64_t cap, const spark_layer_desc *desc,
                                      int B, int T, int hidden, int H, int Hkv, void *y,
                                      void *workspace, size_t workspace_bytes, void *stream) {
    spark_status st = check_hidden(hidden);
    if (st != SPARK_OK) return st;
    const size_t core = spark_attn_prefill_workspace_size(B, T, H, Hkv, desc);
    if (!desc) return SPARK_ERR_NULL;
    if (core == 0) {
        // the core's own checks name the problem
        st = prefill_impl(nullptr, nullptr, nullptr, desc, B, T, H, Hkv, nullptr, nullptr, nullptr,
                          0, nullptr, nullptr, 0, stream, true);
        return st != SPARK_OK ? st : SPARK_ERR_SHAPE;
    }
    if (B == 0 || T == 0) return SPARK_OK;
    if (!x || !w_qkv || !w_g || !w_o || !pos || !y || !workspace) return SPARK_ERR_NULL;
    if ((k_cache == nullptr) != (v_cache == nullptr)) return SPARK_ERR_NULL;
    if (!aligned16(x) || !aligned16(w_qkv) || !aligned16(w_g) || !aligned16(w_o) ||
        !aligned16(y))
        return SPARK_ERR_ALIGN;
    const long long rows = static_cast<long long>(B) * T;
    const LayerPlan pl = plan_layer(core, rows, H, Hkv);
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return SPARK_ERR_ALIGN;
    if (workspace_bytes < pl.bytes) return SPARK_ERR_WORKSPACE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *qkv = ws + pl.qkv, *attn = ws + pl.attn;
    float *gate = reinterpret_cast<float *>(ws + pl.gate);
    // every check of the core call below, before anything is enqueued
    st = prefill_impl(qkv, gate, pos, desc, B, T, H, Hkv, attn, k_cache, v_cache, cap, nullptr,
                      ws, core, stream, true);
    if (st != SPARK_OK) return st;
    st = check_layer_linears(x, w_qkv, w_g, w_o, y, rows, hidden, H, Hkv, ws, pl);
    if (st != SPARK_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (rope_in_projection(rows, desc)) {
        // RoPE in the q_k_v_proj epilogue; the core then rotates nothing
        RopeTable rt;
        fill_rope_table(desc, &rt);
        spark_layer_desc core_desc = *desc;
        core_desc.rot_dim = 0;
        st = project_in(x, w_qkv, w_g, rows, hidden, H, Hkv, ws, pl, s, &rt, pos);
        if (st != SPARK_OK) return st;
        st = prefill_impl(qkv, gate, pos, &core_desc, B, T, H, Hkv, attn, k_cache, v_cache, cap,
                          nullptr, ws, core, stream, false);
    } else {
        st = project_in(x, w_qkv, w_g, rows, hidden, H, Hkv, ws, pl, s);
        if (st != SPARK_OK) return st;
        st = prefill_impl(qkv, gate, pos, desc, B, T, H, Hkv, attn, k_cache, v_cache, cap,
                          nullptr, ws, core, stream, false);
    }
    if (st != SPARK_OK) return st;
    return project_out(attn, w_o, y, rows, hidden, H, ws, s);
}

size_t spark_attn_layer_decode_workspace_size(int B, int hidden, int H, int Hkv, int64_t cap,
                                              const spark_layer_desc *desc) {
    if (check_hidden(hidden) != SPARK_OK) return 0;
    const size_t core = spark_attn_decode_workspace_size(B, H, Hkv, cap, desc);
    if (core == 0) return 0;
    return plan_layer(core, B, H, Hkv).bytes;
}

spark_status spark_attn_layer_decode(const void *x, const void *w_qkv, const void *w_g,
                                     const void *w_o, const int32_t *pos, void *k_cache,
                                     void *v_cache, int64_t cap, const spark_layer_desc *desc,
                                     int B, int hidden, int H, int Hkv, void *y, void *workspace,
                                     size_t workspace_bytes, void *stream) {
    spark_status st = check_hidden(hidden);
    if (st != SPARK_OK) return st;
    if (!desc) return SPARK_ERR_NULL;
    const size_t core = spark_attn_decode_workspace_size(B, H, Hkv, cap, desc);
    if (core == 0) {
        st = decode_impl(nullptr, nullptr, nullptr, nullptr, nullptr, cap, desc, B, H, Hkv,
                         nullptr, nullptr, 0, stream, true);
        return st != SPARK_OK ? st : SPARK_ERR_SHAPE;
    }
    if (B == 0) return SPARK_OK;
    if (!x || !w_qkv || !w_g || !w_o || !pos || !k_cache || !v_cache || !y || !workspace)
        return SPARK_ERR_NULL;
    if (!aligned16(x) || !aligned16(w_qkv) || !aligned16(w_g) || !aligned16(w_o) ||
        !aligned16(y))
        return SPARK_ERR_ALIGN;
    const LayerPlan pl = plan_layer(core, B, H, Hkv);
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return SPARK_ERR_ALIGN;
    if (workspace_bytes < pl.bytes) return SPARK_ERR_WORKSPACE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *qkv = ws + pl.qkv, *attn = ws + pl.attn;
    float *gate = reinterpret_cast<float *>(ws + pl.gate);
    st = decode_impl(qkv, gate, pos, k_cache, v_cache, cap, desc, B, H, Hkv, attn, ws, core,
                     stream, true);
    if (st != SPARK_OK) return st;
    st = check_layer_linears(x, w_qkv, w_g, w_o, y, B, hidden, H, Hkv, ws, pl);
    if (st != SPARK_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = project_in(x, w_qkv, w_g, B, hidden, H, Hkv, ws, pl, s);
    if (st != SPARK_OK) return st;
    st = decode_impl(qkv, gate, pos, k_cache, v_cache, cap, desc, B, H, Hkv, attn, ws, core,
                     stream, false);
    if (st != SPARK_OK) return st;
    return project_out(attn, w_o, y, B, hidden, H, ws, s);
}

}  // extern "C"
