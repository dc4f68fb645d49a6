// common.cuh -- constants, launch parameters and the RoPE angle helper shared
// by the kernels of the attention core.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <utility>

#include "bands.cuh"
#include "ptx.cuh"
#include "rope_math.cuh"

namespace spark {

constexpr int kHeadDim = 256;
constexpr int kMaxRopePairs = kHeadDim / 2;

// log2(e) / sqrt(256): scores are kept in base-2 units, s * kScaleLog2.
constexpr float kScaleLog2 = 1.4426950408889634f / 16.0f;

// Bytes reserved at the start of every workspace for the status word.
constexpr size_t kWorkspaceHeader = 256;

// RoPE frequencies of one layer type, in turns per position:
// u_k = theta^(-2k/r) / (2 pi), stored as an unevaluated fp32 sum hi + lo
// (computed on the host in fp64).
struct RopeTable {
    float2 u[kMaxRopePairs];
    int rot_dim;
};

// cos and sin of the RoPE angle of one pair at an integer position: the
// exact reduction in turns of rope_math.cuh, then sincospif.
__device__ __forceinline__ void rope_cos_sin(int pos, float2 u, float &c, float &s) {
    const float t = rope_turns(pos, u.x, u.y);
    sincospif(__fmul_rn(2.0f, t), &s, &c);
}

// Rotates one (x1, x2) pair: y1 = x1 c - x2 s, y2 = x2 c + x1 s.
__device__ __forceinline__ void rope_rotate(float x1, float x2, float c, float s, float &y1,
                                            float &y2) {
    y1 = __fsub_rn(__fmul_rn(x1, c), __fmul_rn(x2, s));
    y2 = __fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, s));
}

__device__ __forceinline__ float sigmoid_f32(float x) { return 1.0f / (1.0f + expf(-x)); }

// Gate activation of the output gate: sigmoid (mode 0) or silu (mode 1).
__device__ __forceinline__ float gate_act(float x, int mode) {
    const float s = sigmoid_f32(x);
    return mode == 1 ? x * s : s;
}

// Launches `kernel` allowing programmatic dependent launch: it may be
// scheduled before the previous kernel on the stream has finished, and waits
// for it with grid_dep_wait before reading global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- decode

struct DecodeParams {
    const __nv_bfloat16 *qkv;  // [B, (H+2Hkv)*256]
    const float *gate;         // [B, H]
    const int32_t *pos;        // [B]
    __nv_bfloat16 *k_cache;    // [B, Hkv, cap, 256]
    __nv_bfloat16 *v_cache;    // [B, Hkv, cap, 256]
    __nv_bfloat16 *out;        // [B, H*256]
    float *part_ml;            // [B, H, nsplit, 2]: running max (base-2 units), sum
    float *part_o;             // [B, H, nsplit, 256]: unnormalised output
    unsigned *status;          // device status word
    long long cap;             // cache slots per (b, kv head)
    int B, H, Hkv, G;
    int kind, window;
    int gate_mode;             // 0 sigmoid, 1 silu
    int nsplit;                // splits per (b, kv head)
    int chunk;                 // scanned slots per split (multiple of 64)
    // 1: the split kernel merges (no merge kernel).  With several splits per
    // (b, kv head) the CTA that finishes last does it, found by counting the
    // finished splits in counters[b * Hkv + g], which every call leaves at 0.
    int fuse_merge;
    unsigned *counters;        // [B * Hkv] when fuse_merge and nsplit > 1
    RopeTable rope;
};

// Whether a decode call merges inside the split kernel.  One warp per head of
// the finishing CTA walks every split, so this pays only for a few splits
// (rings, short caches): at most kFuseMaxSplits.  With more than one split
// the finished splits are counted in the workspace header, in the words after
// the status word, one per (sequence, KV head); every call leaves them at 0.
constexpr int kFuseMaxSplits = 8;
constexpr int kHeaderCounters = static_cast<int>(kWorkspaceHeader / sizeof(unsigned)) - 1;

inline bool decode_fuses_merge(int nsplit, long long B_times_Hkv, bool have_counters) {
    if (nsplit == 1) return true;
    return have_counters && nsplit <= kFuseMaxSplits && B_times_Hkv <= kHeaderCounters;
}

// ---------------------------------------------------------------- prefill

struct PrefillParams {
    const __nv_bfloat16 *qkv;  // [B, T, (H+2Hkv)*256]
    const float *gate;         // [B, T, H]
    const int32_t *pos;        // [B, T]
    __nv_bfloat16 *krot;       // [B, Hkv, T, rot_w]: rotated leading dims of K
    __nv_bfloat16 *k_cache;    // optional [B, Hkv, cap, 256]: receives rotated K
    __nv_bfloat16 *v_cache;    // optional [B, Hkv, cap, 256]: receives V
    long long cap;             // cache slots (when k_cache is set)
    const int32_t *start;      // optional [B]: tokens cached before this chunk (chunked
                               // prefill: queries and keys are then at start + t)
    unsigned *status;
    int B, T, H, Hkv, G;
    int kind, window;
    int gate_mode;             // 0 sigmoid, 1 silu
    int rot_w;                 // rot_dim rounded up to 64: leading K dims read from krot
    int n_qtiles;              // query tiles per (b, kv head)
    int wave;                  // CTAs resident at once (one per SM): a CTA pulls the
                               // query tile of CTA blockIdx + wave into L2
    int defer_wait;            // nonzero: a library kernel of the same call runs just
                               // before the attention kernel, so only the key/value
                               // loads wait for it (inputs are complete already)
    RopeTable rope;
};

}  // namespace spark
