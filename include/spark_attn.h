/*
 * spark_attn.h -- C ABI of the Spark-X2.5 gated GQA attention core on one
 * GB300 (sm_103a).
 *
 * What the library computes (page titles and sections of the sources):
 *
 *  Spark-X2.5 architecture (4B / 1.7B), §3 "head-wise output gate", Eq. 1:
 *      out = ( softmax(Q K^T / sqrt(256)) V ) * sigmoid(gate_logit)
 *  per query head, the gate being one fp32 scalar per (token, head) that is
 *  broadcast over the head's 256 dims.  Q, K, V come from the fused
 *  q_k_v_proj output, laid out per token as Q (H heads) || K (Hkv heads) ||
 *  V (Hkv heads), 256 bf16 each (same §3: width H*256 + 2*Hkv*256).  Query
 *  head h reads KV head h / (H/Hkv) (grouped-query attention, §1 table).
 *
 *  Same page, §4 "layered RoPE": Q and K are rotated before the product.
 *  For k < r/2, with r = rot_dim and a = pos * theta^(-2k/r):
 *      y_k = x_k cos a - x_{k+r/2} sin a,  y_{k+r/2} = x_{k+r/2} cos a + x_k sin a
 *  dims >= r pass through unchanged (partial RoPE: full_attention layers use
 *  theta 5e6 and r = 64, sliding_attention layers theta 1e4 and r = 256).
 *
 *  Same page, §2 "hybrid attention": full layers are causal (key j visible
 *  from query i iff j <= i); sliding layers add the window, key j visible
 *  iff 0 <= i - j < window (512 in both released models; the window
 *  includes the query itself).
 *
 *  Decode follows the KV-cache behaviour the Spark-X2.5-4B hybrid-attention
 *  explainer (lshu.cn) describes: full layers keep every token, sliding
 *  layers keep only the latest `window` tokens.  Here a full layer's cache is
 *  contiguous (token j at slot j) and a sliding layer's cache is a ring of
 *  `cap` slots (token j at slot j mod cap, cap >= window).  Cached keys are
 *  stored after RoPE.  A step first writes the new token's rotated key and
 *  its value into slot(pos), then attends over the visible tokens.
 *
 * Numerics: bf16 inputs and outputs, fp32 accumulation.  Rotated Q and K are
 * rounded to bf16 once (tensor-core operands), softmax probabilities are
 * rounded to bf16 for the P*V product, the gate multiplies the fp32
 * normalised output and the result is rounded to bf16 (round to nearest even).
 * RoPE angles are reduced exactly in fp32 (positions below 2^24).
 *
 * Conventions for every entry point:
 *  - All data pointers are DEVICE pointers of the current CUDA device (except
 *    the host buffers of spark_attn_prefill_host), 16-byte aligned, dense
 *    row-major in the stated layout.  The caller owns every
 *    buffer; the library allocates no device memory and keeps no per-call
 *    state between calls.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously; nothing synchronizes.
 *  - Argument errors are found on the host before anything is enqueued; the
 *    call then returns the status and leaves every output untouched.
 *  - Faults found on the device (a position outside the cache, a bounded wait
 *    that ran out) set bits in the workspace's status word (see
 *    spark_attn_read_status); the kernels never trap.
 *  - B == 0 (and T == 0 for prefill) is a valid empty call: SPARK_OK, nothing
 *    is enqueued.
 */
#ifndef SPARK_ATTN_H
#define SPARK_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPARK_HEAD_DIM 256

typedef enum spark_status {
    SPARK_OK = 0,
    SPARK_ERR_NULL = 1,        /* a required pointer is NULL */
    SPARK_ERR_SHAPE = 2,       /* a size is negative or inconsistent (H % Hkv, window < 1, ...) */
    SPARK_ERR_UNSUPPORTED = 3, /* valid but not built: H/Hkv not in {1,2,4,8}, rot_dim not a
                                  multiple of 16, gate_mode other than sigmoid or silu */
    SPARK_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned (workspace: 256-byte) */
    SPARK_ERR_CAPACITY = 5,    /* a sliding ring smaller than its window, cap < 1 */
    SPARK_ERR_WORKSPACE = 6,   /* workspace NULL or smaller than the size query returns */
    SPARK_ERR_CUDA = 7,        /* a CUDA call failed while enqueuing (no device, launch error) */
    SPARK_ERR_DEVICE = 8       /* the current device is not an sm_103 GPU */
} spark_status;

typedef enum spark_layer_kind {
    SPARK_LAYER_FULL = 0,      /* causal; contiguous decode cache */
    SPARK_LAYER_SLIDING = 1    /* causal sliding window; ring decode cache */
} spark_layer_kind;

typedef enum spark_gate_mode {
    SPARK_GATE_SIGMOID = 0,    /* out *= 1 / (1 + exp(-g)), g = gate logit (released models) */
    SPARK_GATE_SILU = 1        /* out *= g / (1 + exp(-g)) (gate_attn_act_mode = silu, §3) */
} spark_gate_mode;

/* Layer-type descriptor (the per-layer fields of the model config). */
typedef struct spark_layer_desc {
    int32_t kind;        /* spark_layer_kind */
    int32_t window;      /* SLIDING: window W >= 1; FULL: ignored */
    double rope_theta;   /* RoPE base theta > 0 */
    int32_t rot_dim;     /* rotated dims r: 0 <= r <= 256, multiple of 16 (0 = no RoPE) */
    int32_t gate_mode;   /* spark_gate_mode */
} spark_layer_desc;

/* Bits of the device status word in the workspace. */
#define SPARK_DEVERR_POSITION 0x1u /* a decode position was negative or >= cap (FULL);
                                      that sequence was skipped */
#define SPARK_DEVERR_TIMEOUT 0x2u  /* a bounded on-chip wait ran out; results are invalid */

/*
 * Prefill: attention of T new tokens per sequence over themselves.
 *
 *   qkv   bf16 [B, T, (H + 2*Hkv) * 256]   fused projection, per token Q||K||V
 *   gate  fp32 [B, T, H]                   gate logits
 *   pos   int32 [B, T]                     RoPE positions, 0 <= pos < 2^24
 *   out   bf16 [B, T, H * 256]             gated output, head h at columns h*256..
 *   workspace  >= spark_attn_prefill_workspace_size(...) bytes, 256-byte
 *              aligned, zeroed once before first use (see spark_attn_read_status)
 *
 * The mask is applied on the token index t inside the sequence (query t sees
 * keys t' <= t, and t - t' < window on SLIDING layers); RoPE uses pos.
 * Returns 0 from the size query for invalid arguments.
 */
size_t spark_attn_prefill_workspace_size(int B, int T, int H, int Hkv,
                                         const spark_layer_desc *desc);

spark_status spark_attn_prefill(const void *qkv, const float *gate, const int32_t *pos,
                                const spark_layer_desc *desc, int B, int T, int H, int Hkv,
                                void *out, void *workspace, size_t workspace_bytes,
                                void *stream);

/*
 * Prefill from and to HOST memory.  Computes exactly what spark_attn_prefill
 * computes, for inputs and outputs that live in host memory:
 *
 *   qkv_h, gate_h, pos_h   HOST pointers, layouts as for spark_attn_prefill
 *   out_h                  HOST pointer, bf16 [B, T, H * 256]
 *   workspace  DEVICE, >= spark_attn_prefill_host_workspace_size(...) bytes,
 *              256-byte aligned, zeroed once before first use (its status word
 *              is read with spark_attn_read_status)
 *
 * The batch goes through device staging areas one piece at a time -- a
 * sequence, or a chunk of a longer one (2048 tokens on FULL layers, 3072 on
 * SLIDING layers; processed as a chunked
 * prefill over a device KV cache in the workspace): copy-ins of later pieces
 * and copy-outs of earlier ones run on two copy streams that the library
 * creates per device on first use, while `stream` computes.  Host buffers should be pinned
 * (cudaHostAlloc / cudaHostRegister); pageable memory still works, with
 * copies that do not overlap.  The call returns once everything is enqueued:
 * synchronize `stream` before reading out_h (work enqueued on `stream` after
 * the call is ordered after the last copy-out).  Inputs must stay unchanged
 * until then.  If a CUDA call fails part-way, SPARK_ERR_CUDA is returned
 * and some sequences may have been processed.
 */
size_t spark_attn_prefill_host_workspace_size(int B, int T, int H, int Hkv,
                                              const spark_layer_desc *desc);

spark_status spark_attn_prefill_host(const void *qkv_h, const float *gate_h, const int32_t *pos_h,
                                     const spark_layer_desc *desc, int B, int T, int H, int Hkv,
                                     void *out_h, void *workspace, size_t workspace_bytes,
                                     void *stream);

/*
 * Prefill that also fills the decode cache: computes exactly what
 * spark_attn_prefill computes and stores every token's rotated key (all 256
 * dims) and value in the cache, as the model does while it prefills
 * (past_key_values.update; Spark-X2.5-4B hybrid-attention explainer, lshu.cn).
 *
 *   k_cache, v_cache  bf16 [B, Hkv, cap, 256], written in place.
 *            FULL: token t -> slot t, needs cap >= T.
 *            SLIDING: ring, token t -> slot t mod cap, needs cap >= window;
 *            only the last min(T, cap) tokens are stored (the others would be
 *            overwritten within the same prefill).
 *   Other arguments as for spark_attn_prefill (same workspace size).
 * A spark_attn_decode at pos = T on the same caches continues the sequence.
 */
spark_status spark_attn_prefill_cache(const void *qkv, const float *gate, const int32_t *pos,
                                      void *k_cache, void *v_cache, int64_t cap,
                                      const spark_layer_desc *desc, int B, int T, int H, int Hkv,
                                      void *out, void *workspace, size_t workspace_bytes,
                                      void *stream);

/*
 * Chunked prefill: T more tokens per sequence on top of a cache that already
 * holds the sequence's first start[b] tokens (as spark_attn_prefill_cache or
 * earlier chunks left it).  Query token t of the chunk sits at index
 * start[b] + t; it attends to every cached key and to the chunk's keys under
 * the layer's mask on those indices.  The chunk's rotated keys and values are
 * stored in the cache first (as spark_attn_prefill_cache stores them), so the
 * next chunk or a spark_attn_decode at pos = start[b] + T continues the
 * sequence.
 *
 *   start    int32 [B] (device): tokens already cached per sequence
 *   k_cache, v_cache  bf16 [B, Hkv, cap, 256], updated in place.
 *            FULL: needs start[b] + T <= cap (checked on the device: a
 *            sequence past the end is skipped and SPARK_DEVERR_POSITION set).
 *            SLIDING: a ring with cap >= window + T - 1 (so the chunk's writes
 *            never replace keys its own rows still see) and cap a multiple of
 *            128.
 *   pos      RoPE positions of the chunk's tokens (normally start[b] + t).
 *   Other arguments as for spark_attn_prefill (same workspace size).
 * Cache slots past the chunk that were never written may hold anything; the
 * call clears the few it reads.
 */
spark_status spark_attn_prefill_chunk(const void *qkv, const float *gate, const int32_t *pos,
                                      void *k_cache, void *v_cache, int64_t cap,
                                      const int32_t *start, const spark_layer_desc *desc, int B,
                                      int T, int H, int Hkv, void *out, void *workspace,
                                      size_t workspace_bytes, void *stream);

/*
 * Decode: one new token per sequence.
 *
 *   qkv      bf16 [B, (H + 2*Hkv) * 256]   the new token's fused projection
 *   gate     fp32 [B, H]
 *   pos      int32 [B]   position of the new token = tokens already cached
 *   k_cache, v_cache  bf16 [B, Hkv, cap, 256], updated in place.
 *            FULL: token j at slot j, needs pos < cap (else the sequence is
 *            skipped and SPARK_DEVERR_POSITION is set).
 *            SLIDING: ring, token j at slot j mod cap, needs cap >= window.
 *   out      bf16 [B, H * 256]
 *   workspace >= spark_attn_decode_workspace_size(...) bytes (split-KV
 *            partial softmax states), 256-byte aligned, zeroed once before
 *            first use.  Its first 256 bytes are a header: the status word,
 *            then counters of finished splits, one per (sequence, KV head),
 *            used when a step has at most 8 splits per (sequence, KV head) and
 *            B * Hkv <= 63 (the split kernel then also does the merge).
 *            Every call leaves the counters at 0; do not write into the
 *            header between calls (spark_attn_read_status clears only the
 *            status word).
 * Returns 0 from the size query for invalid arguments.
 */
size_t spark_attn_decode_workspace_size(int B, int H, int Hkv, int64_t cap,
                                        const spark_layer_desc *desc);

spark_status spark_attn_decode(const void *qkv, const float *gate, const int32_t *pos,
                               void *k_cache, void *v_cache, int64_t cap,
                               const spark_layer_desc *desc, int B, int H, int Hkv,
                               void *out, void *workspace, size_t workspace_bytes,
                               void *stream);

/*
 * Number of kernels one spark_attn_decode call with these arguments enqueues
 * on the current device: 2 (the split kernel, then the merge kernel) or 1
 * (the split kernel merges itself: one split per (sequence, KV head), or at
 * most 8 of them with B * Hkv <= 63).  For callers that count or budget
 * launches (CUDA graphs, schedulers).  Returns 0 for invalid arguments and
 * for B == 0.  Host-only: touches no device memory.
 */
int spark_attn_decode_launch_count(int B, int H, int Hkv, int64_t cap,
                                   const spark_layer_desc *desc);

/*
 * Decode without a caller-provided workspace.
 *
 * The paper has no counterpart to this call; it exists for callers that
 * cannot allocate device memory for a workspace: code that runs under a
 * memory manager owning all device memory (a serving runtime with a pool
 * reserved up front, a plugin host that hands over only inputs and outputs),
 * or code on a path where cudaMalloc is not allowed because it synchronizes
 * the device.  It computes exactly what spark_attn_decode computes, with the
 * same arguments except the workspace.  This call allocates nothing.
 *
 *  - Scratch: the split-KV partial states live in one library-owned device
 *    buffer of SPARK_NOALLOC_SCRATCH_BYTES (8 MiB), held by every device that
 *    loads the library until the process exits.  A call that would need more
 *    (spark_attn_decode_workspace_size(...) > SPARK_NOALLOC_SCRATCH_BYTES,
 *    e.g. large batches over long caches) returns SPARK_ERR_WORKSPACE and
 *    enqueues nothing.  The buffer needs no zeroing: each call writes the
 *    partial states it later reads.
 *  - Sharing: all calls on a device share the buffer and it keeps the last
 *    call's contents.  Calls that overlap on the GPU (different streams, or
 *    several host threads without ordering) race on it and give wrong
 *    results; order them on one stream.
 *  - Set-up: the first call on each device looks up the buffer's device
 *    address (cudaGetSymbolAddress, with that device current).  Make that
 *    first call before any stream capture.  The address is kept per device
 *    together with the CUDA context it belongs to; when a later call finds
 *    another context current on the device (the caller reset the device, so
 *    its primary context and the library's module were rebuilt), it looks
 *    the address up again, so that call too should come before any capture.
 *  - device_status: optional DEVICE pointer to a uint32 that receives the
 *    SPARK_DEVERR_* bits (OR-ed in, never cleared by the library); NULL
 *    means those faults are not reported.  A split that gives up on a
 *    bounded wait (SPARK_DEVERR_TIMEOUT) leaves a neutral partial state, so
 *    nothing an earlier call left in the buffer is merged; the output then
 *    lacks that split's keys, and only device_status tells the caller.
 */
#define SPARK_NOALLOC_SCRATCH_BYTES (8u << 20)

spark_status spark_attn_decode_noalloc(const void *qkv, const float *gate, const int32_t *pos,
                                       void *k_cache, void *v_cache, int64_t cap,
                                       const spark_layer_desc *desc, int B, int H, int Hkv,
                                       void *out, uint32_t *device_status, void *stream);

/*
 * The attention block around the core (Spark-X2.5 architecture, §3 Eq. 1 and
 * Fig. 1): q_k_v_proj and g_proj read the normed hidden state x, the core
 * attends, out_proj maps the gated output back to the hidden size:
 *
 *   qkv  = bf16( x W_qkv^T )      W_qkv bf16 [(H + 2*Hkv) * 256, hidden]
 *   g    = bf16( x W_g^T )        W_g   bf16 [H, hidden]   (one logit per head)
 *   a    = core(qkv, g, pos)      as spark_attn_prefill / spark_attn_decode
 *   y    = bf16( a W_o^T )        W_o   bf16 [hidden, H * 256]
 *
 * Weights use the PyTorch Linear layout (out_features x in_features, row
 * major); there are no biases.  Every product accumulates in fp32 and rounds
 * once to bf16 (the checkpoints' dtype, §1); the residual add and the norms
 * stay outside.  With more than 8 rows the projections run on the library's
 * tcgen05 GEMM (spark_attn_linear), q_k_v_proj and g_proj in one launch; with
 * at most 8 (a decode step) on a weight-streaming GEMV, g_proj in the same
 * pass as q_k_v_proj.  hidden must be a positive multiple of 8 (16-byte rows;
 * else SPARK_ERR_UNSUPPORTED).
 *
 * Prefill:
 *   x  bf16 [B, T, hidden];  pos int32 [B, T];  y bf16 [B, T, hidden]
 *   k_cache, v_cache, cap: optional (both NULL, cap ignored) -- when given,
 *            the call also fills the decode cache as spark_attn_prefill_cache
 *            does (same capacity rules).
 * Decode (one new token per sequence):
 *   x  bf16 [B, hidden];  pos int32 [B];  y bf16 [B, hidden]
 *   k_cache, v_cache, cap as for spark_attn_decode (required).
 * workspace: >= the size query's bytes, 256-byte aligned, zeroed once before
 * first use; its status word (spark_attn_read_status) is the core's.  Every
 * argument, including the core's, is checked before anything is enqueued.
 * The size queries return 0 for invalid arguments.
 */
size_t spark_attn_layer_prefill_workspace_size(int B, int T, int hidden, int H, int Hkv,
                                               const spark_layer_desc *desc);

spark_status spark_attn_layer_prefill(const void *x, const void *w_qkv, const void *w_g,
                                      const void *w_o, const int32_t *pos, void *k_cache,
                                      void *v_cache, int64_t cap, const spark_layer_desc *desc,
                                      int B, int T, int hidden, int H, int Hkv, void *y,
                                      void *workspace, size_t workspace_bytes, void *stream);

size_t spark_attn_layer_decode_workspace_size(int B, int hidden, int H, int Hkv, int64_t cap,
                                              const spark_layer_desc *desc);

spark_status spark_attn_layer_decode(const void *x, const void *w_qkv, const void *w_g,
                                     const void *w_o, const int32_t *pos, void *k_cache,
                                     void *v_cache, int64_t cap, const spark_layer_desc *desc,
                                     int B, int hidden, int H, int Hkv, void *y, void *workspace,
                                     size_t workspace_bytes, void *stream);

/*
 * Dense bf16 projection y = x W^T (the Linear layers around the core:
 * Spark-X2.5 architecture, §3 Fig. 1 and §6 -- q_k_v_proj 2560 -> 6144,
 * g_proj 2560 -> 16, out_proj 4096 -> 2560 for the 4B shapes).
 *
 *   x  bf16 [M, K] row major;  W  bf16 [N, K] (PyTorch Linear layout);
 *   y  bf16 [M, N] = round-to-nearest-even of the fp32-accumulated product.
 *
 * Runs on the 5th-generation tensor cores (tcgen05, TMA, accumulators in
 * TMEM), one persistent CTA per SM.  N and K must be multiples of 8 (else
 * SPARK_ERR_UNSUPPORTED); M >= 0 (M == 0 enqueues nothing).  device_status:
 * required DEVICE pointer to a uint32 that receives SPARK_DEVERR_TIMEOUT if a
 * bounded wait ran out (OR-ed in, never cleared by the library).  No scratch
 * memory is used.
 */
spark_status spark_attn_linear(const void *x, const void *w, void *y, int64_t M, int N, int K,
                               uint32_t *device_status, void *stream);

/*
 * Copies the sticky device status word out of a workspace (synchronizes on
 * `stream`).  If `clear` is non-zero the word is reset to 0 afterwards.
 */
spark_status spark_attn_read_status(void *workspace, uint32_t *status_out, int clear,
                                    void *stream);

/* Static description of a status code (never NULL). */
const char *spark_status_str(spark_status status);

/* Library build version, "major.minor.patch". */
const char *spark_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPARK_ATTN_H */
