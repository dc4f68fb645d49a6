// decode.cu -- one decode step of the gated GQA attention core.
//
// Spark-X2.5 architecture (4B / 1.7B), §3 Eq. 1 (softmax(QK^T/16) V times the
// per-head sigmoid gate) and §4 (layered RoPE); the cache behaviour is the one
// the Spark-X2.5-4B hybrid-attention explainer (lshu.cn) describes: full
// layers keep every token, sliding layers only the latest `window`.
//
// One or two kernels on one stream:
//   decode_split_kernel  grid (nsplit, Hkv, B).  Each CTA streams a chunk of
//       cache slots of one (sequence, KV head) through a TMA ring in shared
//       memory and keeps an online softmax for the G query heads of the group
//       (scores and P*V on the tensor cores, keys in the M dimension).  It
//       writes one partial state (running max, sum, unnormalised output) per
//       head.
//   decode_merge_kernel  grid (Hkv, B).  Rotates q and the new key, scores the
//       new token, merges it with the partial states (log-sum-exp rescale),
//       applies the gate, and stores the new key/value at slot(pos).
// When each (sequence, KV head) has one split, or at most kFuseMaxSplits of
// them and B * Hkv fits the counters of the workspace header (rings, short
// caches), the split kernel does the merge itself, with the same arithmetic:
// the CTA that finishes last (a counter of finished splits) merges the
// states, so the step is one launch instead of two.
// The new token is not read from the cache by the split kernel, so the cache
// write can come last without a race: on a full layer slot(pos) lies past
// every cached token, and on a ring it holds token pos - cap, which is out of
// the window (cap >= window).
#include "common.cuh"

namespace spark {

constexpr int kDecTile = 64;                              // cache slots per stage
// TMA stages of a CTA: three for long scans; one where a CTA scans at most
// kDecShortTiles tiles (rings), so that two CTAs fit on an SM and the grid of a
// batch of rings runs as one wave.
constexpr int kDecStagesLong = 3;
constexpr int kDecShortTiles = 8;
constexpr int kDecWarps = 4;                              // consumers, 16 slots each
constexpr int kDecThreads = (kDecWarps + 1) * 32;         // + one producer warp
constexpr int kDecTileBytes = kDecTile * kHeadDim * 2;    // 32 KB (K or V)
constexpr int kDecStageBytes = 2 * kDecTileBytes;         // K + V
constexpr int kDecQBytes = 8 * kHeadDim * 2;              // 8 (padded) query heads
// Kernels that merge: the new token's rotated key and value, and the gate
// logits of the group's (at most 8) heads.
constexpr int kDecNewBytes = 2 * kHeadDim * 2 + 8 * 4;
constexpr int dec_smem_bytes(int stages, bool fuse) {
    return 1024 + stages * kDecStageBytes + kDecQBytes + (fuse ? kDecNewBytes : 0) +
           3 * stages * 8;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Warps per query head in the merge (each takes every S-th split), and the
// largest group the merge kernel's shared reduction buffers hold.
constexpr int kMergeWarps = 4;
constexpr int kMergeMaxG = 8;
__host__ __device__ constexpr int merge_warps(int G) { return G <= 4 ? kMergeWarps : 2; }

// The new token seen by query head h of KV head g: q and the new key rotated
// at pos and rounded to bf16, the score x_new = q.k_new / 16 in base-2 units,
// and this lane's 8 dims of v_new.  Lane l holds dims 8l..8l+7; the rotated
// key is kept packed (bf16) for the cache store.
struct NewToken {
    float x_new;
    float v[8];
    uint32_t kb[4];
    uint4 vv;
};

__device__ __forceinline__ NewToken score_new_token(const DecodeParams &P, int b, int g, int h,
                                                    long long p, int lane) {
    NewToken nt;
    const size_t width = static_cast<size_t>(P.H + 2 * P.Hkv) * kHeadDim;
    const __nv_bfloat16 *row = P.qkv + b * width;
    const uint4 qv = *reinterpret_cast<const uint4 *>(row + static_cast<size_t>(h) * kHeadDim + lane * 8);
    const uint4 kv = *reinterpret_cast<const uint4 *>(row + static_cast<size_t>(P.H + g) * kHeadDim + lane * 8);
    nt.vv = *reinterpret_cast<const uint4 *>(row + static_cast<size_t>(P.H + P.Hkv + g) * kHeadDim + lane * 8);
    const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
    const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w};
    const uint32_t vw[4] = {nt.vv.x, nt.vv.y, nt.vv.z, nt.vv.w};
    float q[8], k[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        q[2 * i] = bf16_lo(qw[i]);
        q[2 * i + 1] = bf16_hi(qw[i]);
        k[2 * i] = bf16_lo(kw[i]);
        k[2 * i + 1] = bf16_hi(kw[i]);
        nt.v[2 * i] = bf16_lo(vw[i]);
        nt.v[2 * i + 1] = bf16_hi(vw[i]);
    }

    // RoPE of this lane's 8 dims d0..d0+7; the partner dims d -/+ r/2 live in
    // the lane r/16 away (r/2 is a multiple of 8).
    const int r = P.rope.rot_dim, half = r / 2, d0 = lane * 8;
    if (r > 0) {
        const int partner = (d0 >= r) ? lane : (d0 < half ? lane + half / 8 : lane - half / 8);
        float qp[8], kp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            qp[i] = __shfl_sync(0xffffffffu, q[i], partner);
            kp[i] = __shfl_sync(0xffffffffu, k[i], partner);
        }
        if (d0 < r) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int kk = (d0 < half) ? d0 + i : d0 + i - half;
                float c, s;
                rope_cos_sin(static_cast<int>(p), P.rope.u[kk], c, s);
                float y1, y2;
                if (d0 < half) {
                    rope_rotate(q[i], qp[i], c, s, y1, y2);
                    q[i] = y1;
                    rope_rotate(k[i], kp[i], c, s, y1, y2);
                    k[i] = y1;
                } else {
                    rope_rotate(qp[i], q[i], c, s, y1, y2);
                    q[i] = y2;
                    rope_rotate(kp[i], k[i], c, s, y1, y2);
                    k[i] = y2;
                }
            }
        }
    }
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        nt.kb[i] = pack_bf16x2(k[2 * i], k[2 * i + 1]);
        const uint32_t qb = pack_bf16x2(q[2 * i], q[2 * i + 1]);
        dot = fmaf(bf16_lo(qb), bf16_lo(nt.kb[i]), dot);
        dot = fmaf(bf16_hi(qb), bf16_hi(nt.kb[i]), dot);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    nt.x_new = dot * kScaleLog2;
    return nt;
}

// The same NewToken from shared memory, where the split kernel's prologue put
// q and the new key rotated and rounded to bf16 (the same values
// score_new_token computes) and the new value: one dot product, no loads from
// global memory.
__device__ __forceinline__ NewToken new_token_from_smem(const __nv_bfloat16 *qs,
                                                        const __nv_bfloat16 *kn,
                                                        const __nv_bfloat16 *vn, int hq,
                                                        int lane) {
    NewToken nt;
    const uint4 qv = *reinterpret_cast<const uint4 *>(qs + hq * kHeadDim + lane * 8);
    const uint4 kv = *reinterpret_cast<const uint4 *>(kn + lane * 8);
    nt.vv = *reinterpret_cast<const uint4 *>(vn + lane * 8);
    const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
    const uint32_t vw[4] = {nt.vv.x, nt.vv.y, nt.vv.z, nt.vv.w};
    nt.kb[0] = kv.x;
    nt.kb[1] = kv.y;
    nt.kb[2] = kv.z;
    nt.kb[3] = kv.w;
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        nt.v[2 * i] = bf16_lo(vw[i]);
        nt.v[2 * i + 1] = bf16_hi(vw[i]);
        dot = fmaf(bf16_lo(qw[i]), bf16_lo(nt.kb[i]), dot);
        dot = fmaf(bf16_hi(qw[i]), bf16_hi(nt.kb[i]), dot);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    nt.x_new = dot * kScaleLog2;
    return nt;
}

// Gated output of head h and, for the first head of the group, the new
// key/value stored at slot(pos) (write-then-attend: no split reads that slot).
__device__ __forceinline__ void store_head(const DecodeParams &P, int b, int g, int hq, int h,
                                           long long p, int d0, const float (&acc)[8], float L,
                                           const NewToken &nt, float gate_logit) {
    const float scale = gate_act(gate_logit, P.gate_mode) / L;
    uint4 ov;
    ov.x = pack_bf16x2(acc[0] * scale, acc[1] * scale);
    ov.y = pack_bf16x2(acc[2] * scale, acc[3] * scale);
    ov.z = pack_bf16x2(acc[4] * scale, acc[5] * scale);
    ov.w = pack_bf16x2(acc[6] * scale, acc[7] * scale);
    *reinterpret_cast<uint4 *>(P.out + static_cast<size_t>(b) * P.H * kHeadDim +
                               static_cast<size_t>(h) * kHeadDim + d0) = ov;
    if (hq == 0) {
        const long long slot = (P.kind == kLayerFull) ? p : p % P.cap;
        const size_t off = ((static_cast<size_t>(b) * P.Hkv + g) * P.cap + slot) * kHeadDim + d0;
        *reinterpret_cast<uint4 *>(P.k_cache + off) = make_uint4(nt.kb[0], nt.kb[1], nt.kb[2], nt.kb[3]);
        *reinterpret_cast<uint4 *>(P.v_cache + off) = nt.vv;
    }
}

// Part sums of the merge for S parts (S = merge_warps(G), a template argument
// so that the prefetched states stay in registers): part q sums the splits
// q, q+S, ..., part 0 starting from the new token, then parts 1..S-1 are
// added to part 0 in turn -- the merge kernel's order, where part q is its
// warp q of the head.
template <int S>
__device__ __forceinline__ void merge_parts(const NewToken &nt, float M, int nvalid,
                                            const float2 (&ml)[kFuseMaxSplits],
                                            const float4 (&pa)[kFuseMaxSplits],
                                            const float4 (&pc)[kFuseMaxSplits], float (&acc)[8],
                                            float &L) {
    const float w_new = fast_exp2(nt.x_new - M);
#pragma unroll
    for (int q = 0; q < S; ++q) {
        const float wq = q == 0 ? w_new : 0.f;
        float Lq = wq, aq[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) aq[i] = nt.v[i] * wq;
#pragma unroll
        for (int sp = q; sp < kFuseMaxSplits; sp += S) {
            if (sp < nvalid) {
                const float w = (ml[sp].x == -INFINITY) ? 0.f : fast_exp2(ml[sp].x - M);
                Lq += ml[sp].y * w;
                aq[0] += pa[sp].x * w;
                aq[1] += pa[sp].y * w;
                aq[2] += pa[sp].z * w;
                aq[3] += pa[sp].w * w;
                aq[4] += pc[sp].x * w;
                aq[5] += pc[sp].y * w;
                aq[6] += pc[sp].z * w;
                aq[7] += pc[sp].w * w;
            }
        }
        if (q == 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = aq[i];
            L = Lq;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] += aq[i];
            L += Lq;
        }
    }
}

// The merge of query head hq of the group, done by one warp of the split
// kernel, with the same arithmetic in the same order as the merge kernel.
// `nt` (the new token) was loaded before the split count; the states of all
// (at most kFuseMaxSplits) splits are then fetched at once.  Other CTAs wrote
// them, so they are read at L2 (ld.global.cg).
__device__ __forceinline__ void merge_head_in_split(const DecodeParams &P, int b, int g, int hq,
                                                    long long p, int nvalid, int lane,
                                                    const NewToken &nt, float gate_logit) {
    const int h = g * P.G + hq, d0 = lane * 8;
    const size_t part0 = (static_cast<size_t>(b) * P.H + h) * P.nsplit;
    float2 ml[kFuseMaxSplits];
    float4 pa[kFuseMaxSplits], pc[kFuseMaxSplits];
#pragma unroll
    for (int sp = 0; sp < kFuseMaxSplits; ++sp) {
        if (sp < nvalid) {
            ml[sp] = __ldcg(reinterpret_cast<const float2 *>(P.part_ml + 2 * (part0 + sp)));
            const float4 *po = reinterpret_cast<const float4 *>(P.part_o + (part0 + sp) * kHeadDim + d0);
            pa[sp] = __ldcg(po);
            pc[sp] = __ldcg(po + 1);
        } else {
            ml[sp] = make_float2(-INFINITY, 0.f);
            pa[sp] = pc[sp] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    // the maximum over the new token and every split (absent ones are -inf)
    float M = nt.x_new;
#pragma unroll
    for (int sp = 0; sp < kFuseMaxSplits; ++sp) M = fmaxf(M, ml[sp].x);
    float acc[8], L;
    if (merge_warps(P.G) == kMergeWarps)
        merge_parts<kMergeWarps>(nt, M, nvalid, ml, pa, pc, acc, L);
    else
        merge_parts<2>(nt, M, nvalid, ml, pa, pc, acc, L);
    store_head(P, b, g, hq, h, p, d0, acc, L, nt, gate_logit);
}

// The same merge where the scan has one split: that split's state is the
// CTA's own, still in shared memory (the per-warp maxima, sums and rescaled
// outputs of the final reduction), so it is summed there in the order the
// global partial state would have been, with no round trip through L2.  A
// CTA that gave up on a wait merges a neutral state.
__device__ __forceinline__ void merge_head_local(const DecodeParams &P, int b, int g, int hq,
                                                 long long p, int lane, const NewToken &nt,
                                                 float gate_logit, const float *red_o,
                                                 const float (&red_m)[kDecWarps][8],
                                                 const float (&red_l)[kDecWarps][8],
                                                 bool aborted) {
    const int h = g * P.G + hq, d0 = lane * 8;
    float2 ml[kFuseMaxSplits];
    float4 pa[kFuseMaxSplits], pc[kFuseMaxSplits];
#pragma unroll
    for (int sp = 0; sp < kFuseMaxSplits; ++sp) {
        ml[sp] = make_float2(-INFINITY, 0.f);
        pa[sp] = pc[sp] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (!aborted) {
        float M = red_m[0][hq];
#pragma unroll
        for (int w = 1; w < kDecWarps; ++w) M = fmaxf(M, red_m[w][hq]);
        float L = 0.f;
        if (M != -INFINITY)
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) L += red_l[w][hq] * fast_exp2(red_m[w][hq] - M);
        ml[0] = make_float2(M, L);
        float o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float a = 0.f;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) a += red_o[(w * 8 + hq) * kHeadDim + d0 + i];
            o[i] = a;
        }
        pa[0] = make_float4(o[0], o[1], o[2], o[3]);
        pc[0] = make_float4(o[4], o[5], o[6], o[7]);
    }
    float M = nt.x_new;
#pragma unroll
    for (int sp = 0; sp < kFuseMaxSplits; ++sp) M = fmaxf(M, ml[sp].x);
    float acc[8], L;
    if (merge_warps(P.G) == kMergeWarps)
        merge_parts<kMergeWarps>(nt, M, 1, ml, pa, pc, acc, L);
    else
        merge_parts<2>(nt, M, 1, ml, pa, pc, acc, L);
    store_head(P, b, g, hq, h, p, d0, acc, L, nt, gate_logit);
}

// kFuse: this CTA's grid merges itself (P.fuse_merge); a separate
// instantiation, so that the kernel of the long scans carries none of it.
template <int kDecStages, bool kFuse>
__global__ void __launch_bounds__(kDecThreads, kDecStages == 1 ? 2 : 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ DecodeParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *stages = smem;
    __nv_bfloat16 *qs = reinterpret_cast<__nv_bfloat16 *>(smem + kDecStages * kDecStageBytes);
    // (kernels that merge) the new token's key, rotated, its value and the gates
    __nv_bfloat16 *kn = qs + 8 * kHeadDim;
    __nv_bfloat16 *vn = kn + kHeadDim;
    float *gq = reinterpret_cast<float *>(vn + kHeadDim);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kDecStages * kDecStageBytes + kDecQBytes +
                                                  (kFuse ? kDecNewBytes : 0));
    uint64_t *empty = full + kDecStages;
    // K and V of a stage land on separate barriers: the scores and the softmax
    // of a tile run while its V is still arriving
    uint64_t *fullv = empty + kDecStages;
    __shared__ int abort_flag;
    __shared__ float red_m[kDecWarps][8];
    __shared__ float red_l[kDecWarps][8];

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    grid_dep_wait();  // inputs and cache may come from the previous kernel
    const long long c_lo = static_cast<long long>(split) * P.chunk;

    // one tile of K and V into stage t % kDecStages
    auto issue_tile = [&](int t) {
        const int s = t % kDecStages;
        const int key0 = static_cast<int>(c_lo + static_cast<long long>(t) * kDecTile);
        uint8_t *kt = stages + s * kDecStageBytes;
        mbar_arrive_expect_tx(&full[s], kDecTileBytes);
#pragma unroll
        for (int c = 0; c < 4; ++c)
            tma_load_4d(kt + c * (kDecTileBytes / 4), &tm_k, &full[s], c * 64, key0, g, b);
        mbar_arrive_expect_tx(&fullv[s], kDecTileBytes);
#pragma unroll
        for (int c = 0; c < 4; ++c)
            tma_load_4d(kt + kDecTileBytes + c * (kDecTileBytes / 4), &tm_v, &fullv[s], c * 64,
                        key0, g, b);
    };
    auto init_stages = [&]() {
        for (int s = 0; s < kDecStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&fullv[s], 1);
            mbar_init(&empty[s], kDecWarps);
        }
        fence_mbar_init();
        abort_flag = 0;
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    };
    // The one-stage kernels (short scans: every CTA of a batch of rings starts
    // at once) load their first tile before the position is read, so the
    // position's latency overlaps the copy.  A split's first slots always lie
    // inside the cache (chunk * split < the longest scan <= cap); a CTA that
    // turns out to have no work waits for the copy to land before it exits.
    constexpr bool kSpeculate = kDecStages == 1;
    const bool producer = tid == kDecWarps * 32;
    if (kSpeculate && producer) {
        init_stages();
        issue_tile(0);
    }

    const long long p = P.pos[b];
    const bool bad_pos = p < 0 || (P.kind == kLayerFull && p >= P.cap);
    // Scanned slots: full layer -> tokens [0, pos); ring -> slots [0, min(pos, cap)).
    const long long n_scan = bad_pos ? 0 : decode_scan_slots(P.kind, p, P.cap);
    const long long c_hi = (c_lo + P.chunk < n_scan) ? c_lo + P.chunk : n_scan;
    if (bad_pos || c_lo >= c_hi) {
        if (bad_pos && split == 0 && g == 0 && tid == 0) atomicOr(P.status, kErrPosition);
        // An empty split: the merge does not read it.  With nothing cached yet
        // no split has work, and a fused merge then comes from split 0, on the
        // new token alone.
        if (kFuse && !bad_pos && n_scan == 0 && split == 0 && warp < kDecWarps)
            for (int hq = warp; hq < P.G; hq += kDecWarps)
                merge_head_in_split(P, b, g, hq, p, 0, lane,
                                    score_new_token(P, b, g, g * P.G + hq, p, lane),
                                    P.gate[static_cast<size_t>(b) * P.H + g * P.G + hq]);
        if (kSpeculate && producer) {
            mbar_wait_plain(&full[0], 0);
            mbar_wait_plain(&fullv[0], 0);
        }
        return;
    }
    const int ntiles = static_cast<int>((c_hi - c_lo + kDecTile - 1) / kDecTile);

    // The producer sets the stages up and starts the first loads at once: they
    // do not depend on the query prologue below, which they overlap.
    const int n_pre = ntiles < kDecStages ? ntiles : kDecStages;
    if (!kSpeculate && producer) {
        init_stages();
        for (int t = 0; t < n_pre; ++t) issue_tile(t);
    }

    // The group's G query heads, rotated and rounded to bf16 (heads G..7 zero).
    const size_t width = static_cast<size_t>(P.H + 2 * P.Hkv) * kHeadDim;
    for (int i = tid; i < 8 * (kHeadDim / 8); i += kDecThreads) {
        const int hh = i / (kHeadDim / 8), v = i % (kHeadDim / 8);
        uint4 val = make_uint4(0, 0, 0, 0);
        if (hh < P.G)
            val = *reinterpret_cast<const uint4 *>(
                P.qkv + b * width + static_cast<size_t>(g * P.G + hh) * kHeadDim + v * 8);
        *reinterpret_cast<uint4 *>(qs + hh * kHeadDim + v * 8) = val;
    }
    if constexpr (kFuse) {
        // the new token for the merge at the end, loaded with q
        if (tid < 2 * (kHeadDim / 8)) {
            const int which = tid / (kHeadDim / 8), v = tid % (kHeadDim / 8);
            const uint4 val = *reinterpret_cast<const uint4 *>(
                P.qkv + b * width + static_cast<size_t>(P.H + which * P.Hkv + g) * kHeadDim + v * 8);
            *reinterpret_cast<uint4 *>((which ? vn : kn) + v * 8) = val;
        } else if (tid < 2 * (kHeadDim / 8) + P.G) {
            const int hh = tid - 2 * (kHeadDim / 8);
            gq[hh] = P.gate[static_cast<size_t>(b) * P.H + g * P.G + hh];
        }
    }
    __syncthreads();
    const int half = P.rope.rot_dim / 2;
    for (int k = tid; k < half; k += kDecThreads) {
        float c, s;
        rope_cos_sin(static_cast<int>(p), P.rope.u[k], c, s);
        for (int hh = 0; hh < P.G; ++hh) {
            const float x1 = __bfloat162float(qs[hh * kHeadDim + k]);
            const float x2 = __bfloat162float(qs[hh * kHeadDim + k + half]);
            float y1, y2;
            rope_rotate(x1, x2, c, s, y1, y2);
            qs[hh * kHeadDim + k] = __float2bfloat16_rn(y1);
            qs[hh * kHeadDim + k + half] = __float2bfloat16_rn(y2);
        }
        if constexpr (kFuse) {
            const float x1 = __bfloat162float(kn[k]);
            const float x2 = __bfloat162float(kn[k + half]);
            float y1, y2;
            rope_rotate(x1, x2, c, s, y1, y2);
            kn[k] = __float2bfloat16_rn(y1);
            kn[k + half] = __float2bfloat16_rn(y2);
        }
    }
    __syncthreads();

    if (warp == kDecWarps) {
        // ------------------------------------------------------ TMA producer
        int issued = n_pre;
        if (lane == 0) {
            for (int t = n_pre; t < ntiles; ++t) {
                if (!mbar_wait(&empty[t % kDecStages], ((t / kDecStages) - 1) & 1, &abort_flag,
                               P.status))
                    break;
                issue_tile(t);
                ++issued;
            }
        }
        __syncwarp();
        __syncthreads();
        // Copies still in flight after an abort must land before the CTA
        // releases its shared memory.
        if (lane == 0 && abort_flag) {
            const int first = issued > kDecStages ? issued - kDecStages : 0;
            for (int t = first; t < issued; ++t) {
                mbar_wait_plain(&full[t % kDecStages], (t / kDecStages) & 1);
                mbar_wait_plain(&fullv[t % kDecStages], (t / kDecStages) & 1);
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    // Q^T as the B operand of S^T = K Q^T: one (b0, b1) pair per 16 dims.
    uint32_t qf[16][2];
    {
        const uint32_t qbase = smem_u32(qs);
#pragma unroll
        for (int ks = 0; ks < 16; ks += 2) {
            const uint32_t addr = qbase + (lane & 7) * (kHeadDim * 2) +
                                  (ks * 16 + (lane >> 3) * 8) * 2;
            ldmatrix_x4(addr, qf[ks][0], qf[ks][1], qf[ks + 1][0], qf[ks + 1][1]);
        }
    }

    float o[16][4];
#pragma unroll
    for (int db = 0; db < 16; ++db) o[db][0] = o[db][1] = o[db][2] = o[db][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const int arow = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;  // K rows (ldmatrix)
    const int vrow = warp * 16 + (lane & 7) + (lane >> 4) * 8;        // V rows (ldmatrix.trans)

    for (int t = 0; t < ntiles; ++t) {
        const int s = t % kDecStages;
        if (!mbar_wait(&full[s], (t / kDecStages) & 1, &abort_flag, P.status)) break;
        const uint32_t kt = smem_u32(stages + s * kDecStageBytes);
        const uint32_t vt = kt + kDecTileBytes;

        // S^T (16 slots x 8 heads) = K (16 x 256) Q^T (256 x 8)
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
            const int gran = ((ks * 16) & 63) / 8 + (lane >> 4);
            const uint32_t addr = kt + (ks >> 2) * (kDecTileBytes / 4) + arow * 128 +
                                  ((gran ^ (arow & 7)) << 4);
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4(addr, a0, a1, a2, a3);
            mma_bf16_16816(sc, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
        }

        // this thread's two slots (rows lane/4 and lane/4 + 8) and two heads
        const long long sa = c_lo + static_cast<long long>(t) * kDecTile + warp * 16 + (lane >> 2);
        const long long sb = sa + 8;
        bool va = sa < c_hi, vb = sb < c_hi;
        if (P.kind == kLayerSliding) {
            va = va && ring_slot_visible(sa, p, P.cap, P.window);
            vb = vb && ring_slot_visible(sb, p, P.cap, P.window);
        }
        const float x0 = va ? sc[0] * kScaleLog2 : -INFINITY;
        const float x1 = va ? sc[1] * kScaleLog2 : -INFINITY;
        const float x2 = vb ? sc[2] * kScaleLog2 : -INFINITY;
        const float x3 = vb ? sc[3] * kScaleLog2 : -INFINITY;
        float t0 = fmaxf(x0, x2), t1 = fmaxf(x1, x3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, off));
            t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, off));
        }
        const float n0 = fmaxf(m0, t0), n1 = fmaxf(m1, t1);
        const float r0 = (n0 == -INFINITY) ? 1.f : fast_exp2(m0 - n0);
        const float r1 = (n1 == -INFINITY) ? 1.f : fast_exp2(m1 - n1);
        const float z0 = (n0 == -INFINITY) ? 0.f : n0;
        const float z1 = (n1 == -INFINITY) ? 0.f : n1;
        const float p0 = fast_exp2(x0 - z0), p1 = fast_exp2(x1 - z1);
        const float p2 = fast_exp2(x2 - z0), p3 = fast_exp2(x3 - z1);
        l0 = l0 * r0 + p0 + p2;
        l1 = l1 * r1 + p1 + p3;
        m0 = n0;
        m1 = n1;
#pragma unroll
        for (int db = 0; db < 16; ++db) {
            o[db][0] *= r0;
            o[db][1] *= r1;
            o[db][2] *= r0;
            o[db][3] *= r1;
        }
        // P^T as the B operand of O^T += V^T P^T (transpose of the score fragment)
        const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p0, p1));
        const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p2, p3));
        if (!mbar_wait(&fullv[s], (t / kDecStages) & 1, &abort_flag, P.status)) break;

        // Slots past the chunk end may hold anything (even NaN bit patterns in
        // a cache that was never written there); their probabilities are 0,
        // but 0 * NaN is NaN in P*V, so this warp zeroes its V rows past the end.
        {
            const long long row0 = c_lo + static_cast<long long>(t) * kDecTile + warp * 16;
            if (row0 + 16 > c_hi) {
                uint8_t *vrows = stages + s * kDecStageBytes + kDecTileBytes;
                for (int rr = 0; rr < 16; ++rr) {
                    if (row0 + rr < c_hi) continue;
                    const int vr = warp * 16 + rr;  // 4 chunks of 128 bytes per row
                    *reinterpret_cast<uint4 *>(vrows + (lane >> 3) * (kDecTileBytes / 4) +
                                               vr * 128 + (lane & 7) * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                // the stage is refilled by TMA later: order these writes first
                fence_proxy_async_smem();
                __syncwarp();
            }
        }
#pragma unroll
        for (int db = 0; db < 16; ++db) {
            const int gran = ((db * 16) & 63) / 8 + ((lane >> 3) & 1);
            const uint32_t addr = vt + (db >> 2) * (kDecTileBytes / 4) + vrow * 128 +
                                  ((gran ^ (vrow & 7)) << 4);
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4_trans(addr, a0, a1, a2, a3);
            mma_bf16_16816(o[db], a0, a1, a2, a3, pb0, pb1);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }

    grid_dep_launch();  // the merge kernel may start its set-up
    // row sums over the 8 lanes that share this thread's heads
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    const int h0 = 2 * (lane & 3), h1 = h0 + 1;
    if (lane < 4) {
        red_m[warp][h0] = m0;
        red_m[warp][h1] = m1;
        red_l[warp][h0] = l0;
        red_l[warp][h1] = l1;
    }
    named_bar_sync(1, kDecWarps * 32);
    // With one split per (sequence, KV head) a merging kernel merges from the
    // reduction buffers in shared memory; no partial state goes to global memory.
    const bool local_merge = kFuse && P.nsplit == 1;
    // abort_flag is stable here: it is only raised inside a wait, and every
    // wait of the producer and the consumers has returned.
    if (!abort_flag) {
        float M0 = red_m[0][h0], M1 = red_m[0][h1];
#pragma unroll
        for (int w = 1; w < kDecWarps; ++w) {
            M0 = fmaxf(M0, red_m[w][h0]);
            M1 = fmaxf(M1, red_m[w][h1]);
        }
        const float s0 = (M0 == -INFINITY) ? 0.f : fast_exp2(m0 - M0);
        const float s1 = (M1 == -INFINITY) ? 0.f : fast_exp2(m1 - M1);
        // every stage has been consumed: the ring is free for the reduction
        float *red_o = reinterpret_cast<float *>(stages);
#pragma unroll
        for (int db = 0; db < 16; ++db) {
            const int d = db * 16 + (lane >> 2);
            // only the group's G heads are read back (heads G..7 are padding)
            if (h0 < P.G) {
                red_o[(warp * 8 + h0) * kHeadDim + d] = o[db][0] * s0;
                red_o[(warp * 8 + h0) * kHeadDim + d + 8] = o[db][2] * s0;
            }
            if (h1 < P.G) {
                red_o[(warp * 8 + h1) * kHeadDim + d] = o[db][1] * s1;
                red_o[(warp * 8 + h1) * kHeadDim + d + 8] = o[db][3] * s1;
            }
        }
        named_bar_sync(1, kDecWarps * 32);
        const size_t part0 = (static_cast<size_t>(b) * P.H + static_cast<size_t>(g) * P.G) * P.nsplit;
        for (int i = tid; !local_merge && i < P.G * kHeadDim; i += kDecWarps * 32) {
            const int hh = i / kHeadDim, d = i % kHeadDim;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) acc += red_o[(w * 8 + hh) * kHeadDim + d];
            P.part_o[(part0 + static_cast<size_t>(hh) * P.nsplit + split) * kHeadDim + d] = acc;
        }
        if (!local_merge && tid < P.G) {
            const int hh = tid;
            float M = red_m[0][hh];
            for (int w = 1; w < kDecWarps; ++w) M = fmaxf(M, red_m[w][hh]);
            float L = 0.f;
            if (M != -INFINITY)
                for (int w = 0; w < kDecWarps; ++w) L += red_l[w][hh] * fast_exp2(red_m[w][hh] - M);
            float2 ml = make_float2(M, L);
            *reinterpret_cast<float2 *>(P.part_ml + 2 * (part0 + static_cast<size_t>(hh) * P.nsplit +
                                                         split)) = ml;
        }
    } else if (!local_merge) {
        // A wait gave up (the status word says so): leave a neutral state
        // (max -inf, sum 0, output 0), which the merge weighs by 0, so that
        // it never merges what an earlier call left in a shared buffer.
        const size_t part0 = (static_cast<size_t>(b) * P.H + static_cast<size_t>(g) * P.G) * P.nsplit;
        for (int i = tid; i < P.G * kHeadDim; i += kDecWarps * 32) {
            const int hh = i / kHeadDim, d = i % kHeadDim;
            P.part_o[(part0 + static_cast<size_t>(hh) * P.nsplit + split) * kHeadDim + d] = 0.f;
        }
        if (tid < P.G)
            *reinterpret_cast<float2 *>(P.part_ml + 2 * (part0 + static_cast<size_t>(tid) * P.nsplit +
                                                         split)) = make_float2(-INFINITY, 0.f);
    }
    if constexpr (!kFuse) {
        __syncthreads();
        return;
    }
    __syncthreads();  // the producer warp has returned after this barrier

    // ---------------------------------------------------------- fused merge
    // Every non-empty split counts itself once it has written its states (an
    // aborted one too, so the count always completes and returns to 0); the
    // one that completes the count merges.  No thread waits on another CTA.
    const int nvalid = static_cast<int>((n_scan + P.chunk - 1) / P.chunk);
    // The new token of this warp's heads (warp, warp + 4), from the copy the
    // prologue staged in shared memory.
    NewToken nt[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int hq = warp + i * kDecWarps;
        if (hq < P.G) nt[i] = new_token_from_smem(qs, kn, vn, hq, lane);
    }
    if (nvalid > 1) {
        __shared__ int last_cta;
        __threadfence();  // this thread's states are visible on the device before the count
        named_bar_sync(1, kDecWarps * 32);
        if (tid == 0) {
            unsigned *cnt = P.counters + static_cast<size_t>(b) * P.Hkv + g;
            last_cta = atomicAdd(cnt, 1u) == static_cast<unsigned>(nvalid - 1);
            if (last_cta) atomicExch(cnt, 0u);  // every split has counted: reset for the next call
        }
        named_bar_sync(1, kDecWarps * 32);
        if (!last_cta) return;
        __threadfence();  // order the reads of the other splits' states after the count
    }
    if (local_merge) {
        const float *red_o = reinterpret_cast<const float *>(stages);
        const bool aborted = abort_flag != 0;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int hq = warp + i * kDecWarps;
            if (hq < P.G)
                merge_head_local(P, b, g, hq, p, lane, nt[i], gq[hq], red_o, red_m, red_l,
                                 aborted);
        }
        return;
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int hq = warp + i * kDecWarps;
        if (hq < P.G) merge_head_in_split(P, b, g, hq, p, nvalid, lane, nt[i], gq[hq]);
    }
}

__global__ void __launch_bounds__(512) decode_merge_kernel(const __grid_constant__ DecodeParams P) {
    __shared__ float red_acc[kMergeMaxG][kMergeWarps - 1][kHeadDim];
    __shared__ float red_l[kMergeMaxG][kMergeWarps - 1];
    const int g = blockIdx.x, b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = static_cast<int>(blockDim.x) / (32 * P.G);  // warps per head
    const int hq = warp / S, part = warp % S;  // head within the group, split phase
    const int h = g * P.G + hq;
    // The new token's q, k and v are inputs of the split kernel, which waited
    // for them before letting this kernel start: rotate and score the token
    // while the split kernel still runs.
    const long long p = P.pos[b];
    if (p < 0 || (P.kind == kLayerFull && p >= P.cap)) {
        if (g == 0 && threadIdx.x == 0) atomicOr(P.status, kErrPosition);
        return;
    }
    const NewToken nt = score_new_token(P, b, g, h, p, lane);
    const float x_new = nt.x_new;
    const float *v = nt.v;
    const int d0 = lane * 8;

    grid_dep_wait();  // partial states of the split kernel
    grid_dep_launch();

    // merge the new token with the partial states of the non-empty splits:
    // the maximum lane-parallel, then the weighted sums, the S warps of a head
    // on interleaved splits with several in flight each
    const long long n_scan = decode_scan_slots(P.kind, p, P.cap);
    const int nvalid = static_cast<int>((n_scan + P.chunk - 1) / P.chunk);
    const size_t part0 = (static_cast<size_t>(b) * P.H + h) * P.nsplit;
    float M = x_new;
    for (int sp = lane; sp < nvalid; sp += 32) M = fmaxf(M, P.part_ml[2 * (part0 + sp)]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float w_new = part == 0 ? fast_exp2(x_new - M) : 0.f;
    float L = w_new;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = v[i] * w_new;
#pragma unroll 4
    for (int sp = part; sp < nvalid; sp += S) {
        const float2 ml = *reinterpret_cast<const float2 *>(P.part_ml + 2 * (part0 + sp));
        const float w = (ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - M);
        L += ml.y * w;
        const float4 *po = reinterpret_cast<const float4 *>(P.part_o + (part0 + sp) * kHeadDim + d0);
        const float4 a = po[0], c = po[1];
        acc[0] += a.x * w;
        acc[1] += a.y * w;
        acc[2] += a.z * w;
        acc[3] += a.w * w;
        acc[4] += c.x * w;
        acc[5] += c.y * w;
        acc[6] += c.z * w;
        acc[7] += c.w * w;
    }
    if (part > 0) {
        float4 *dst = reinterpret_cast<float4 *>(&red_acc[hq][part - 1][d0]);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        if (lane == 0) red_l[hq][part - 1] = L;
    }
    __syncthreads();
    if (part > 0) return;
    for (int w = 0; w + 1 < S; ++w) {
        const float4 *src = reinterpret_cast<const float4 *>(&red_acc[hq][w][d0]);
        const float4 a = src[0], c = src[1];
        acc[0] += a.x;
        acc[1] += a.y;
        acc[2] += a.z;
        acc[3] += a.w;
        acc[4] += c.x;
        acc[5] += c.y;
        acc[6] += c.z;
        acc[7] += c.w;
        L += red_l[hq][w];
    }
    store_head(P, b, g, hq, h, p, d0, acc, L, nt, P.gate[static_cast<size_t>(b) * P.H + h]);
}

// ---------------------------------------------------------------- launchers

cudaError_t launch_decode(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const DecodeParams &P,
                          cudaStream_t stream) {
    const bool short_scan = P.chunk <= kDecShortTiles * kDecTile;
    auto kernel = short_scan ? (P.fuse_merge ? decode_split_kernel<1, true>
                                             : decode_split_kernel<1, false>)
                             : (P.fuse_merge ? decode_split_kernel<kDecStagesLong, true>
                                             : decode_split_kernel<kDecStagesLong, false>);
    const int smem = dec_smem_bytes(short_scan ? 1 : kDecStagesLong, P.fuse_merge != 0);
    cudaError_t err =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    dim3 grid(P.nsplit, P.Hkv, P.B);
    err = launch_overlapped(kernel, grid, dim3(kDecThreads), smem, stream, tm_k, tm_v, P);
    if (err != cudaSuccess || P.fuse_merge) return err;
    return launch_overlapped(decode_merge_kernel, dim3(P.Hkv, P.B),
                             dim3(32 * P.G * merge_warps(P.G)), 0, stream, P);
}

}  // namespace spark
