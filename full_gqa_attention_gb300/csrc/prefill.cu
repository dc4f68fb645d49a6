// prefill.cu -- prefill of the gated GQA attention core on the 5th-generation
// tensor cores (tcgen05, accumulators in TMEM, operands staged by TMA).
//
// Spark-X2.5 architecture (4B / 1.7B): §3 Eq. 1 (softmax(QK^T/16) V times the
// per-head sigmoid gate), §4 layered RoPE, §2 causal / sliding-window masks.
//
// Two kernels on one stream:
//   prefill_rope_k_kernel  writes the leading rot_w = roundup(rot_dim, 64)
//       dims of every key, rotated, to a workspace [B][Hkv][T][rot_w].  The
//       other key dims and all of V are read by TMA straight from qkv.
//   prefill_attn_kernel    one CTA per (query tile, KV head, sequence).  A
//       query tile is 128 rows = (128/G) tokens x the G query heads that share
//       the KV head, so every K/V byte brought on chip serves all G heads.
//       Warp roles:
//         warp 0       TMA producer (Q tile once, then K and V through a ring
//                      of 16 KB slots)
//         warp 1       TMEM owner and QK^T issuer (one thread)
//         warp 2       P*V issuer (one thread)
//         warps 4..11  softmax, two warpgroups: query row i (TMEM lane i) is
//                      shared by thread i of each; warpgroup w owns score
//                      columns [64w, 64w+64) and output dims [128w, 128w+128)
//       TMEM (512 columns): O [128 x 256 fp32] in columns 0..255, two score
//       buffers S0/S1 [128 x 128 fp32] in 256..383 and 384..511.  The
//       probabilities P (bf16 pairs) overwrite columns 0..31 (keys 0..63) and
//       64..95 (keys 64..127) of their score buffer, each warpgroup inside the
//       columns it read, and feed P*V as the TMEM A operand.  QK^T of tile j+1 runs on
//       the tensor cores while the softmax of tile j runs on the CUDA cores.
//       Q is rotated in shared memory by the softmax threads (each its own
//       row) before the first product.  Key tiles wholly outside the causal
//       band / window are never visited; boundary tiles are masked per element.
//       Online softmax in base 2 with a lazy rescale: the reference maximum
//       moves only when a row's maximum grows by more than 2^8.
#include "common.cuh"

namespace spark {

// ---------------------------------------------------------------- K RoPE

constexpr int kRopeThreads = 256;

__global__ void __launch_bounds__(kRopeThreads) prefill_rope_k_kernel(
    const __grid_constant__ PrefillParams P) {
    const int r = P.rope.rot_dim, half = r / 2;
    const int n_rot = half / 8;              // groups of 8 rotated pairs
    const int n_copy = (P.rot_w - r) / 8;    // groups of 8 dims copied unrotated
    const int items = n_rot + n_copy;
    grid_dep_wait();  // qkv and pos may come from the previous kernel
    grid_dep_launch();
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long row = idx / items;
    const int it = static_cast<int>(idx % items);
    if (row >= static_cast<long long>(P.B) * P.T) return;
    const int b = static_cast<int>(row / P.T), t = static_cast<int>(row % P.T);
    const size_t width = static_cast<size_t>(P.H + 2 * P.Hkv) * kHeadDim;
    const __nv_bfloat16 *src = P.qkv + row * width + static_cast<size_t>(P.H) * kHeadDim;
    __nv_bfloat16 *dst0 = P.krot + (static_cast<size_t>(b) * P.Hkv * P.T + t) * P.rot_w;
    const size_t head_stride = static_cast<size_t>(P.T) * P.rot_w;
    if (it < n_rot) {
        const int k0 = it * 8;
        const int p = P.pos[row];
        float c[8], s[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rope_cos_sin(p, P.rope.u[k0 + i], c[i], s[i]);
        for (int g = 0; g < P.Hkv; ++g) {
            const uint4 a = *reinterpret_cast<const uint4 *>(src + g * kHeadDim + k0);
            const uint4 bb = *reinterpret_cast<const uint4 *>(src + g * kHeadDim + k0 + half);
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
            const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
            uint32_t ya[4], yb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float y1l, y2l, y1h, y2h;
                rope_rotate(bf16_lo(aw[i]), bf16_lo(bw[i]), c[2 * i], s[2 * i], y1l, y2l);
                rope_rotate(bf16_hi(aw[i]), bf16_hi(bw[i]), c[2 * i + 1], s[2 * i + 1], y1h, y2h);
                ya[i] = pack_bf16x2(y1l, y1h);
                yb[i] = pack_bf16x2(y2l, y2h);
            }
            __nv_bfloat16 *dst = dst0 + g * head_stride;
            *reinterpret_cast<uint4 *>(dst + k0) = make_uint4(ya[0], ya[1], ya[2], ya[3]);
            *reinterpret_cast<uint4 *>(dst + k0 + half) = make_uint4(yb[0], yb[1], yb[2], yb[3]);
        }
    } else {
        const int d0 = r + (it - n_rot) * 8;
        for (int g = 0; g < P.Hkv; ++g)
            *reinterpret_cast<uint4 *>(dst0 + g * head_stride + d0) =
                *reinterpret_cast<const uint4 *>(src + g * kHeadDim + d0);
    }
}

// ---------------------------------------------------------------- KV cache fill

// Stores every token's rotated K (all 256 dims) and its V in the decode cache,
// the step a model takes while it prefills (past_key_values.update): token t
// goes to slot t of a full layer's cache, or to slot t mod cap of a sliding
// layer's ring, where only the last cap tokens survive.  One thread per
// (token, group of 8 rotated pairs / 8 copied K dims / 8 V dims), looping over
// KV heads so each angle is computed once per (token, pair).
__global__ void __launch_bounds__(kRopeThreads) prefill_store_kv_kernel(
    const __grid_constant__ PrefillParams P) {
    grid_dep_wait();
    grid_dep_launch();
    const int r = P.rope.rot_dim, half = r / 2;
    const int n_rot = half / 8, n_kcopy = (kHeadDim - r) / 8, n_v = kHeadDim / 8;
    const int items = n_rot + n_kcopy + n_v;
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long row = idx / items;
    const int it = static_cast<int>(idx % items);
    if (row >= static_cast<long long>(P.B) * P.T) return;
    const int b = static_cast<int>(row / P.T), t = static_cast<int>(row % P.T);
    if (P.kind == kLayerSliding && t < P.T - P.cap) return;  // overwritten later in the ring
    const long long a = (P.start ? static_cast<long long>(P.start[b]) : 0) + t;  // absolute index
    if (a < 0 || (P.kind == kLayerFull && a >= P.cap)) {
        if (it == 0 && t == 0) atomicOr(P.status, kErrPosition);
        return;
    }
    const long long slot = (P.kind == kLayerFull) ? a : a % P.cap;
    const size_t width = static_cast<size_t>(P.H + 2 * P.Hkv) * kHeadDim;
    const __nv_bfloat16 *src_k = P.qkv + row * width + static_cast<size_t>(P.H) * kHeadDim;
    const __nv_bfloat16 *src_v = src_k + static_cast<size_t>(P.Hkv) * kHeadDim;
    const size_t head_stride = static_cast<size_t>(P.cap) * kHeadDim;
    const size_t base = (static_cast<size_t>(b) * P.Hkv * P.cap + slot) * kHeadDim;
    if (it < n_rot) {
        const int k0 = it * 8;
        const int p = P.pos[row];
        float c[8], s[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rope_cos_sin(p, P.rope.u[k0 + i], c[i], s[i]);
        for (int g = 0; g < P.Hkv; ++g) {
            const uint4 a = *reinterpret_cast<const uint4 *>(src_k + g * kHeadDim + k0);
            const uint4 bb = *reinterpret_cast<const uint4 *>(src_k + g * kHeadDim + k0 + half);
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
            const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
            uint32_t ya[4], yb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float y1l, y2l, y1h, y2h;
                rope_rotate(bf16_lo(aw[i]), bf16_lo(bw[i]), c[2 * i], s[2 * i], y1l, y2l);
                rope_rotate(bf16_hi(aw[i]), bf16_hi(bw[i]), c[2 * i + 1], s[2 * i + 1], y1h, y2h);
                ya[i] = pack_bf16x2(y1l, y1h);
                yb[i] = pack_bf16x2(y2l, y2h);
            }
            __nv_bfloat16 *dst = P.k_cache + base + g * head_stride;
            *reinterpret_cast<uint4 *>(dst + k0) = make_uint4(ya[0], ya[1], ya[2], ya[3]);
            *reinterpret_cast<uint4 *>(dst + k0 + half) = make_uint4(yb[0], yb[1], yb[2], yb[3]);
        }
    } else if (it < n_rot + n_kcopy) {
        const int d0 = r + (it - n_rot) * 8;
        for (int g = 0; g < P.Hkv; ++g)
            *reinterpret_cast<uint4 *>(P.k_cache + base + g * head_stride + d0) =
                *reinterpret_cast<const uint4 *>(src_k + g * kHeadDim + d0);
    } else {
        const int d0 = (it - n_rot - n_kcopy) * 8;
        for (int g = 0; g < P.Hkv; ++g)
            *reinterpret_cast<uint4 *>(P.v_cache + base + g * head_stride + d0) =
                *reinterpret_cast<const uint4 *>(src_v + g * kHeadDim + d0);
    }
}

// Zeroes the cache slots that the last key tile of a chunked prefill may read
// past the chunk end but that no token has written yet (a full layer's future
// slots, or ring slots on the first pass): their probabilities are 0, but a
// never-written slot may hold NaN bit patterns and 0 * NaN is NaN in P*V.
// One block per sequence.
__global__ void __launch_bounds__(kRopeThreads) cache_zero_tail_kernel(
    const __grid_constant__ PrefillParams P) {
    grid_dep_wait();
    grid_dep_launch();
    const int b = blockIdx.x;
    if (P.start[b] < 0) return;  // flagged by the store kernel
    const long long a_end = static_cast<long long>(P.start[b]) + P.T;
    const long long a_stop = (a_end + 127) / 128 * 128;
    const long long last = a_stop < P.cap ? a_stop : P.cap;  // slots a_end..last-1
    const int per_slot = P.Hkv * (kHeadDim / 8);             // 16-byte words per slot and tensor
    for (long long w = threadIdx.x; w < (last - a_end) * per_slot; w += blockDim.x) {
        const long long j = a_end + w / per_slot;
        const int g = static_cast<int>((w % per_slot) / (kHeadDim / 8));
        const int d0 = static_cast<int>(w % (kHeadDim / 8)) * 8;
        const size_t off = ((static_cast<size_t>(b) * P.Hkv + g) * P.cap + j) * kHeadDim + d0;
        *reinterpret_cast<uint4 *>(P.k_cache + off) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(P.v_cache + off) = make_uint4(0, 0, 0, 0);
    }
}

// ---------------------------------------------------------------- attention

constexpr int kBM = 128;                  // query rows per tile
constexpr int kBN = 128;                  // keys per tile
constexpr int kSlotBytes = 16384;         // ring slot: 128 keys x 64 dims (K) or 32 keys x 256 (V)
constexpr int kSlots = 8;
constexpr int kQBytes = 4 * kSlotBytes;   // 128 rows x 256 dims, as 4 chunks of 64 dims
constexpr int kAttnThreads = 384;
constexpr int kPrefetchMaxTiles = 8;      // CTAs this short pull the next wave's Q into L2
constexpr int kSoftmaxWarp0 = 4;
constexpr int kSoftmaxThreads = 256;        // two warpgroups, 64 score columns each
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256;

// barriers
constexpr int kBarQFull = 0;
constexpr int kBarQReady = 1;
constexpr int kBarSlotFull = 2;                 // kSlots of them
constexpr int kBarSlotEmpty = 2 + kSlots;       // kSlots of them
constexpr int kBarSFull = 2 + 2 * kSlots;       // 2
constexpr int kBarPReady = 4 + 2 * kSlots;      // 2
constexpr int kBarODone = 6 + 2 * kSlots;
constexpr int kBarMmaDrain = 7 + 2 * kSlots;
constexpr int kBarOFinal = 8 + 2 * kSlots;      // every P*V done (one phase per CTA)
constexpr int kBarMaxX = 9 + 2 * kSlots;        // 2: half-row maxima exchanged (per tile parity)
constexpr int kNumBars = 11 + 2 * kSlots;

constexpr int kAttnSmemBytes = 1024 + kQBytes + kSlots * kSlotBytes + 256;

constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, 0, 0);        // Q, K both K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, kHeadDim, 0, 1);   // V is N(=dim)-major

// Byte offset of 16-byte granule `gran` (0..31 across the 256 dims) of row
// `row` inside a tile stored as 4 chunks of [rows][64 dims] with the 128-byte
// TMA swizzle (granule index XOR row mod 8 inside each 1024-byte atom).
__device__ __forceinline__ uint32_t sw128_offset(int row, int gran) {
    return static_cast<uint32_t>((gran >> 3) * kSlotBytes + row * 128 +
                                 (((gran & 7) ^ (row & 7)) << 4));
}

// RoPE of one query row held in shared memory (the 128-byte-swizzled Q tile),
// for the pair groups of warpgroup `wg`.  The G lanes holding the G heads of
// one token compute 8/G of the 8 angles of a group each and exchange them by
// shuffles, so each angle is computed once per token.
template <int G>
__device__ __forceinline__ void rotate_q_row(uint8_t *qbuf, int row, int lane, int wg, int pos,
                                             const RopeTable &rope) {
    const int half = rope.rot_dim / 2;
    const int base = lane & ~(G - 1), sub = lane & (G - 1);
    for (int k0 = wg * 8; k0 < half; k0 += 16) {
        float cw[8 / G], sw[8 / G];
#pragma unroll
        for (int m = 0; m < 8 / G; ++m) rope_cos_sin(pos, rope.u[k0 + sub + G * m], cw[m], sw[m]);
        float c[8], s[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            c[i] = __shfl_sync(0xffffffffu, cw[i / G], base + (i % G));
            s[i] = __shfl_sync(0xffffffffu, sw[i / G], base + (i % G));
        }
        uint4 *pa = reinterpret_cast<uint4 *>(qbuf + sw128_offset(row, k0 / 8));
        uint4 *pb = reinterpret_cast<uint4 *>(qbuf + sw128_offset(row, (k0 + half) / 8));
        const uint4 a = *pa, bb = *pb;
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
        const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
        uint32_t ya[4], yb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float y1l, y2l, y1h, y2h;
            rope_rotate(bf16_lo(aw[i]), bf16_lo(bw[i]), c[2 * i], s[2 * i], y1l, y2l);
            rope_rotate(bf16_hi(aw[i]), bf16_hi(bw[i]), c[2 * i + 1], s[2 * i + 1], y1h, y2h);
            ya[i] = pack_bf16x2(y1l, y1h);
            yb[i] = pack_bf16x2(y2l, y2h);
        }
        *pa = make_uint4(ya[0], ya[1], ya[2], ya[3]);
        *pb = make_uint4(yb[0], yb[1], yb[2], yb[3]);
    }
}

__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Where the keys and values come from: the fused projection (one-shot
// prefill), or the KV cache of a chunked prefill -- a full layer's, one slot
// per token, or a sliding layer's ring.  In a chunked prefill the queries are
// chunk tokens at absolute index start[b] + t, the cache already holds this
// chunk's keys and values, and tm_kv_k / tm_kv_v map the caches.  Each source
// is its own instantiation, so that no kernel carries another's addressing
// (the ring's slot arithmetic would sit in every inlined load of the
// producer).
enum KvSource : int { kKvFromQkv = 0, kKvFromCache = 1, kKvFromRing = 2 };

// The layer kind is a template argument too, so that a kernel carries no
// arithmetic of the other kind; kKindAny reads it from P.kind instead.  Which
// instantiation serves which layer was chosen by timing: the kind-specialised
// builds are faster for both chunked kinds and the one-shot sliding layer,
// the generic one for the one-shot full layer.
constexpr int kKindAny = -1;

// kG: the GQA group size when fixed at compile time (the Spark-X2.5 shapes
// all use 4), 0 to read it from P.G.  Timing chose the fixed size for the
// sliding-kind kernels only; the full-kind ones measured faster without it.
template <int kSrc, int kKind, int kG>
__global__ void __launch_bounds__(kAttnThreads, 1)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_kv_k,
                        const __grid_constant__ CUtensorMap tm_kv_v,
                        const __grid_constant__ CUtensorMap tm_krot,
                        const __grid_constant__ CUtensorMap tm_out,
                        const __grid_constant__ PrefillParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *qbuf = smem;
    uint8_t *ring = smem + kQBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + kSlots * kSlotBytes);
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    __shared__ float red_max[2][2][kBM];   // [tile parity][warpgroup][row]: half-row maxima
    __shared__ float red_l[2][kBM];        // [warpgroup][row]: half-row sums

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kind = kKind == kKindAny ? P.kind : kKind;
    const int G = kG > 0 ? kG : P.G, tq = kBM / G;
    const int units = P.Hkv * P.B;
    const int qtile = P.n_qtiles - 1 - static_cast<int>(blockIdx.x) / units;  // longest first
    const int rem = static_cast<int>(blockIdx.x) % units;
    const int g = rem % P.Hkv, b = rem / P.Hkv;
    const int t0 = qtile * tq;
    const int t_end = (t0 + tq < P.T) ? t0 + tq : P.T;  // exclusive

    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            uint32_t count = 1;
            if (i == kBarQReady || i == kBarPReady || i == kBarPReady + 1 || i == kBarMaxX ||
                i == kBarMaxX + 1)
                count = kSoftmaxThreads;
            if (i == kBarMmaDrain) count = 2;  // one commit from each MMA issuer
            mbar_init(&bars[i], count);
        }
        fence_mbar_init();
        abort_flag = 0;
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base_sh, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_kv_k);
        tma_prefetch_desc(&tm_kv_v);
        if (P.rot_w > 0) tma_prefetch_desc(&tm_krot);
        tma_prefetch_desc(&tm_out);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    // Programmatic dependent launch.  The kernel before this one may still run.
    // When it is one of this call's own (rotated K, or the chunk's cache store),
    // it waited for the call's inputs before letting this kernel start, so only
    // the producer waits, before its first key/value load.  Otherwise every
    // thread waits here, before reading any input.
    if (!P.defer_wait) grid_dep_wait();

    // Absolute indices: queries t0..t_end-1 of the chunk sit at start + t.
    int start = 0;
    bool skip = false;
    if constexpr (kSrc != kKvFromQkv) {
        start = P.start[b];
        skip = start < 0 || (kind == kLayerFull && static_cast<long long>(start) + P.T > P.cap);
        if (skip && tid == 0 && qtile == P.n_qtiles - 1 && g == 0) atomicOr(P.status, kErrPosition);
    }
    const int a0 = start + t0;
    // a ring is read in 128-key tiles aligned to its 128-slot boundaries, so
    // that no tile wraps around the end of the ring
    const KeyTiles kt = prefill_key_tiles(kind, P.window, a0, start + t_end, kBN,
                                          kSrc == kKvFromRing);
    const int kv_lo = kt.kv_lo;
    const int ntiles = skip ? 0 : kt.ntiles;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        int sc = 0;  // ring slots filled so far
        if (lane == 0 && !skip) {
            mbar_arrive_expect_tx(&bars[kBarQFull], kQBytes);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tma_load_4d(qbuf + c * kSlotBytes, &tm_q, &bars[kBarQFull], c * 64, g * G, t0, b);
            // the CTA one wave later (likely the next one on this SM) finds its
            // query tile in L2 -- when this CTA is short (a sliding layer's, or
            // the last waves of a causal one); behind a long CTA the tile would
            // be evicted before use and read twice
            const long long nb = static_cast<long long>(blockIdx.x) + P.wave;
            if (P.wave > 0 && nb < gridDim.x && ntiles <= kPrefetchMaxTiles) {
                const int nq = P.n_qtiles - 1 - static_cast<int>(nb / units);
                const int nrem = static_cast<int>(nb % units);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    tma_prefetch_l2_4d(&tm_q, c * 64, (nrem % P.Hkv) * G, nq * tq, nrem / P.Hkv);
            }
            if (P.defer_wait) grid_dep_wait();  // rotated K / the cache are ready
            bool ok = true;
            auto next_slot = [&](int &slot) -> bool {
                slot = sc % kSlots;
                if (sc >= kSlots &&
                    !mbar_wait(&bars[kBarSlotEmpty + slot], ((sc / kSlots) - 1) & 1, &abort_flag,
                               P.status))
                    return false;
                mbar_arrive_expect_tx(&bars[kBarSlotFull + slot], kSlotBytes);
                return true;
            };
            auto load_k = [&](int j) -> bool {
                const int key0 = kv_lo + j * kBN;
                for (int c = 0; c < 4; ++c) {
                    int slot;
                    if (!next_slot(slot)) return false;
                    uint8_t *dst = ring + slot * kSlotBytes;
                    if constexpr (kSrc != kKvFromQkv) {
                        const int slot0 =
                            kSrc == kKvFromRing ? key0 % static_cast<int>(P.cap) : key0;
                        tma_load_4d(dst, &tm_kv_k, &bars[kBarSlotFull + slot], c * 64, slot0, g,
                                    b);
                    } else if (c * 64 < P.rot_w) {
                        tma_load_3d(dst, &tm_krot, &bars[kBarSlotFull + slot], c * 64, key0,
                                    b * P.Hkv + g);
                    } else {
                        tma_load_4d(dst, &tm_kv_k, &bars[kBarSlotFull + slot], c * 64, P.H + g,
                                    key0, b);
                    }
                    ++sc;
                }
                return true;
            };
            auto load_v = [&](int j) -> bool {
                const int key0 = kv_lo + j * kBN;
                for (int vs = 0; vs < 4; ++vs) {
                    int slot;
                    if (!next_slot(slot)) return false;
                    uint8_t *dst = ring + slot * kSlotBytes;
                    if constexpr (kSrc != kKvFromQkv) {
                        const int slot0 =
                            kSrc == kKvFromRing ? key0 % static_cast<int>(P.cap) : key0;
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            tma_load_4d(dst + c * (kSlotBytes / 4), &tm_kv_v,
                                        &bars[kBarSlotFull + slot], c * 64, slot0 + vs * 32, g, b);
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            tma_load_4d(dst + c * (kSlotBytes / 4), &tm_kv_v,
                                        &bars[kBarSlotFull + slot], c * 64, P.H + P.Hkv + g,
                                        key0 + vs * 32, b);
                    }
                    ++sc;
                }
                return true;
            };
            ok = load_k(0);
            if (ok && ntiles > 1) ok = load_k(1);
            for (int j = 0; ok && j < ntiles; ++j) {
                ok = load_v(j);
                if (ok && j + 2 < ntiles) ok = load_k(j + 2);
            }
        }
        __syncwarp();
        tc_fence_before();
        __syncthreads();
        // after an abort, copies in flight must land before shared memory is released
        if (lane == 0 && abort_flag) {
            mbar_wait_plain(&bars[kBarQFull], 0);
            const int first = sc > kSlots ? sc - kSlots : 0;
            for (int s = first; s < sc; ++s)
                mbar_wait_plain(&bars[kBarSlotFull + (s % kSlots)], (s / kSlots) & 1);
        }
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------ MMA issuers
        // Two threads issue the products: warp 1's lane 0 the QK^T of every
        // key tile, warp 2's lane 0 every P*V, so neither waits for the
        // other's issue.  Both replay the producer's load order (K0, K1, then
        // per tile j: V_j, K_{j+2}) to find the ring slots of their chunks.
        // The barriers carry the dependencies between them: P*V of tile j
        // waits for P_j (softmax), and QK^T of tile j+2, which overwrites the
        // score buffer holding P_j, waits for P*V of tile j to complete.
        const bool qk_role = warp == 1;
        if (lane == 0 && !skip) {
            // Shared-memory descriptors built once: the address field holds
            // (address mod 2^18) / 16 in its low bits, and every operand lies
            // below 2^18, so an operand at byte offset o from a base has the
            // base's descriptor plus o / 16.  This keeps the issue loop short.
            const uint64_t q_desc = smem_desc_sw128(smem_u32(qbuf), 16, 1024);
            const uint64_t k_desc = smem_desc_sw128(smem_u32(ring), 16, 1024);
            const uint64_t v_desc = smem_desc_sw128(smem_u32(ring), kSlotBytes / 4, 1024);
            // (the full-layer cache instance measured faster building each
            // descriptor in place)
            constexpr bool kDescInPlace = kSrc == kKvFromCache;
            const uint32_t q_addr = smem_u32(qbuf), ring_addr = smem_u32(ring);
            int sc = 0;  // ring slots of the producer's loads before the next one
            bool ok = true;
            auto mma_qk = [&](int j) -> bool {
                const uint32_t d = tmem + kColS + (j & 1) * kBN;
                for (int c = 0; c < 4; ++c) {
                    const int slot = sc % kSlots;
                    if (!mbar_wait(&bars[kBarSlotFull + slot], (sc / kSlots) & 1, &abort_flag,
                                   P.status))
                        return false;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad =
                            kDescInPlace
                                ? smem_desc_sw128(q_addr + c * kSlotBytes + kk * 32, 16, 1024)
                                : q_desc + static_cast<uint32_t>((c * kSlotBytes + kk * 32) >> 4);
                        const uint64_t bd =
                            kDescInPlace
                                ? smem_desc_sw128(ring_addr + slot * kSlotBytes + kk * 32, 16, 1024)
                                : k_desc + static_cast<uint32_t>((slot * kSlotBytes + kk * 32) >> 4);
                        mma_ss(d, ad, bd, kIdescQK, (c | kk) != 0);
                    }
                    tc_commit(&bars[kBarSlotEmpty + slot]);
                    ++sc;
                }
                tc_commit(&bars[kBarSFull + (j & 1)]);
                return true;
            };
            auto mma_pv = [&](int j) -> bool {
                const uint32_t pcol = tmem + kColS + (j & 1) * kBN;
                for (int vs = 0; vs < 4; ++vs) {
                    const int slot = sc % kSlots;
                    if (!mbar_wait(&bars[kBarSlotFull + slot], (sc / kSlots) & 1, &abort_flag,
                                   P.status))
                        return false;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const int ks = vs * 2 + kk;  // 16-key step within the tile
                        const uint64_t bd =
                            kDescInPlace
                                ? smem_desc_sw128(ring_addr + slot * kSlotBytes + kk * 2048,
                                                  kSlotBytes / 4, 1024)
                                : v_desc + static_cast<uint32_t>((slot * kSlotBytes + kk * 2048) >> 4);
                        // P of keys 0..63 sits in packed columns 0..31, keys 64..127 in 64..95
                        const uint32_t acol = pcol + (ks < 4 ? ks * 8 : 64 + (ks - 4) * 8);
                        mma_ts(tmem + kColO, acol, bd, kIdescPV, (j > 0 || ks > 0));
                    }
                    tc_commit(&bars[kBarSlotEmpty + slot]);
                    ++sc;
                }
                tc_commit(&bars[kBarODone]);
                return true;
            };
            if (qk_role) {
                ok = mbar_wait(&bars[kBarQReady], 0, &abort_flag, P.status);
                tc_fence_after();
                if (ok) ok = mma_qk(0);
                if (ok && ntiles > 1) ok = mma_qk(1);
                for (int j = 0; ok && j < ntiles; ++j) {
                    sc += 4;  // V_j: the other issuer's
                    if (j + 2 < ntiles) {
                        // QK^T of tile j+2 overwrites the score buffer whose
                        // first half holds P_j: wait until P*V of tile j
                        // (accumulator O) has finished reading it.  P*V of tile
                        // j+1 needs QK^T of tile j+1, issued before this wait,
                        // so the barrier is never two phases ahead of it.
                        ok = mbar_wait(&bars[kBarODone], j & 1, &abort_flag, P.status);
                        if (ok) {
                            tc_fence_after();
                            ok = mma_qk(j + 2);
                        }
                    }
                }
            } else {
                sc = ntiles > 1 ? 8 : 4;  // after K0 and K1
                for (int j = 0; ok && j < ntiles; ++j) {
                    ok = mbar_wait(&bars[kBarPReady + (j & 1)], (j >> 1) & 1, &abort_flag,
                                   P.status);
                    if (!ok) break;
                    tc_fence_after();
                    ok = mma_pv(j);
                    if (j + 2 < ntiles) sc += 4;  // K_{j+2}: the other issuer's
                }
                // The epilogue waits on a barrier of its own: a parity wait on
                // kBarODone could be two phases behind when the last softmax
                // tile finishes before P*V of the tile before it.
                if (ok) tc_commit(&bars[kBarOFinal]);
            }
            // every product either thread issued must finish before TMEM is
            // released (the drain barrier counts one arrival from each)
            tc_commit(&bars[kBarMmaDrain]);
            mbar_wait_plain(&bars[kBarMmaDrain], 0);
        }
        __syncwarp();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (qk_role) tmem_dealloc(tmem, kTmemCols);
    } else if (warp >= kSoftmaxWarp0) {
        // ------------------------------------------------------ softmax
        const int wq = warp & 3;                        // TMEM lane quarter of this warp
        const int wg = (warp - kSoftmaxWarp0) >> 2;     // warpgroup: score-column half
        const int row = wq * 32 + lane;                 // TMEM lane, query row
        const int sth = tid - kSoftmaxWarp0 * 32;       // 0..255 among softmax threads
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        const int tok = t0 + row / G;
        const int tok_abs = start + tok;                // absolute index for the mask
        const int head = g * G + row % G;
        const bool valid = tok < P.T;
        const size_t trow = static_cast<size_t>(b) * P.T + (valid ? tok : 0);
        const int p = valid ? P.pos[trow] : 0;
        const float gate_logit = valid ? P.gate[trow * P.H + head] : 0.f;
        bool ok = !skip && mbar_wait(&bars[kBarQFull], 0, &abort_flag, P.status);

        // rotate this row of Q in place (bf16 in, fp32 math, bf16 out); the
        // two warpgroups take alternate groups of 8 pairs, and the G rows of a
        // token (adjacent lanes) share the angles
        if (ok) {
            if constexpr (kG > 0) {
                rotate_q_row<kG>(qbuf, row, lane, wg, p, P.rope);
            } else {
                switch (G) {
                    case 1: rotate_q_row<1>(qbuf, row, lane, wg, p, P.rope); break;
                    case 2: rotate_q_row<2>(qbuf, row, lane, wg, p, P.rope); break;
                    case 4: rotate_q_row<4>(qbuf, row, lane, wg, p, P.rope); break;
                    default: rotate_q_row<8>(qbuf, row, lane, wg, p, P.rope); break;
                }
            }
        }
        fence_proxy_async_smem();
        if (!skip) mbar_arrive(&bars[kBarQReady]);

        // Scores stay in raw units s = q.k; probabilities are
        // exp2(s * kScaleLog2 - m * kScaleLog2) with m the row's reference max.
        // The reference moves only when the row max grows past it by the
        // raw equivalent of 2^8.
        constexpr float kLazyRaw = 8.0f / kScaleLog2;
        const int a_last = start + t_end - 1;
        const int col0 = wg * 64;                       // first score column of this thread
        float m_run = -INFINITY, l_part = 0.f;
        for (int j = 0; ok && j < ntiles; ++j) {
            ok = mbar_wait(&bars[kBarSFull + (j & 1)], (j >> 1) & 1, &abort_flag, P.status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t sbase = lane_base + kColS + (j & 1) * kBN;
            uint32_t sv[64];
            tmem_ld32(sbase + col0, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
            tmem_ld32(sbase + col0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
            tmem_ld_wait();
            float x[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) x[c] = __uint_as_float(sv[c]);
            const int key0 = kv_lo + j * kBN;
            if (tile_needs_mask(kind, P.window, key0, kBN, a0, a_last)) {
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const bool vis = key_visible(kind, P.window, tok_abs, key0 + col0 + c);
                    x[c] = vis ? x[c] : -INFINITY;
                }
            }
            // row max of this half (8 independent chains), then of the row
            float m8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) m8[i] = x[i];
#pragma unroll
            for (int c = 8; c < 64; ++c) m8[c & 7] = fmaxf(m8[c & 7], x[c]);
            const float mloc = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                     fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
            // exchange with the other half of the row (a bounded wait, so a
            // warp that gave up elsewhere cannot strand the others)
            red_max[j & 1][wg][row] = mloc;
            mbar_arrive(&bars[kBarMaxX + (j & 1)]);
            ok = mbar_wait(&bars[kBarMaxX + (j & 1)], (j >> 1) & 1, &abort_flag, P.status);
            if (!ok) break;
            const float m_new = fmaxf(mloc, red_max[j & 1][wg ^ 1][row]);

            // tcgen05.ld/st are warp-collective: the O rescale runs for the
            // whole warp (alpha is 1 on rows that keep their reference)
            const bool bump = m_new > m_run + kLazyRaw;
            const bool rescale_row = bump && m_run != -INFINITY;
            const float alpha = rescale_row ? fast_exp2((m_run - m_new) * kScaleLog2) : 1.f;
            if (bump) {
                l_part *= alpha;
                m_run = m_new;
            }
            if (j > 0 && __any_sync(0xffffffffu, rescale_row)) {
                ok = mbar_wait(&bars[kBarODone], (j - 1) & 1, &abort_flag, P.status);
                if (!ok) break;
                tc_fence_after();
                for (int c = wg * 128; c < wg * 128 + 128; c += 32) {
                    uint32_t ov[32];
                    tmem_ld32(lane_base + kColO + c, ov);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                    tmem_st32(lane_base + kColO + c, ov);
                }
            }
            const float neg = (m_run == -INFINITY) ? 0.f : -m_run * kScaleLog2;
            uint32_t pk[32];
            float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float p0 = fast_exp2(fmaf(x[2 * c], kScaleLog2, neg));
                const float p1 = fast_exp2(fmaf(x[2 * c + 1], kScaleLog2, neg));
                l8[c & 7] += p0 + p1;
                pk[c] = pack_bf16x2(p0, p1);
            }
            l_part += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
            tmem_st32(sbase + wg * 64, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bars[kBarPReady + (j & 1)]);
        }

        // epilogue: O / l * sigmoid(gate) -> bf16 -> staged in the Q buffer -> TMA store
        if (sth == 0) grid_dep_launch();
        if (ok) ok = mbar_wait(&bars[kBarOFinal], 0, &abort_flag, P.status);
        if (skip) ok = false;
        red_l[wg][row] = l_part;
        named_bar(1, kSoftmaxThreads);
        {
            // every softmax thread runs this block (barrier counts must match);
            // only the store below depends on the abort flag
            tc_fence_after();
            const float l_row = l_part + red_l[wg ^ 1][row];
            const float scale = valid ? gate_act(gate_logit, P.gate_mode) / l_row : 0.f;
            // two 32-column loads in flight per wait (the loads' latency overlaps)
            for (int c = wg * 128; c < wg * 128 + 128; c += 64) {
                uint32_t ov[2][32];
                tmem_ld32(lane_base + kColO + c, ov[0]);
                tmem_ld32(lane_base + kColO + c + 32, ov[1]);
                tmem_ld_wait();
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(ov[h][8 * q + 0]) * scale,
                                          __uint_as_float(ov[h][8 * q + 1]) * scale);
                        w.y = pack_bf16x2(__uint_as_float(ov[h][8 * q + 2]) * scale,
                                          __uint_as_float(ov[h][8 * q + 3]) * scale);
                        w.z = pack_bf16x2(__uint_as_float(ov[h][8 * q + 4]) * scale,
                                          __uint_as_float(ov[h][8 * q + 5]) * scale);
                        w.w = pack_bf16x2(__uint_as_float(ov[h][8 * q + 6]) * scale,
                                          __uint_as_float(ov[h][8 * q + 7]) * scale);
                        *reinterpret_cast<uint4 *>(qbuf + sw128_offset(row, (c + 32 * h) / 8 + q)) = w;
                    }
            }
            fence_proxy_async_smem();
            named_bar(1, kSoftmaxThreads);
            if (sth == 0 && !abort_flag && !skip) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    tma_store_4d(&tm_out, qbuf + c * kSlotBytes, c * 64, g * G, t0, b);
                tma_store_commit();
                tma_store_wait_read();  // the staging buffer is read; the writes land by grid end
            }
        }
        tc_fence_before();
        __syncthreads();
    } else {
        // warp 3 has no role
        __syncthreads();
    }
}

// ---------------------------------------------------------------- launcher

// The attention kernel for a KV source and layer kind; sliding-kind kernels
// are specialised for a group of 4.
template <int kSrc, int kKind>
auto attn_kernel_for(int G) {
    if constexpr (kKind == kLayerSliding)
        return G == 4 ? prefill_attn_kernel<kSrc, kKind, 4> : prefill_attn_kernel<kSrc, kKind, 0>;
    else
        return prefill_attn_kernel<kSrc, kKind, 0>;
}

cudaError_t launch_prefill(const CUtensorMap &tm_q, const CUtensorMap &tm_kv_k,
                           const CUtensorMap &tm_kv_v, const CUtensorMap &tm_krot,
                           const CUtensorMap &tm_out, const PrefillParams &P_in,
                           cudaStream_t stream) {
    PrefillParams P = P_in;
    // a library kernel runs before the attention kernel on every path but the
    // one-shot prefill without rotated dims
    P.defer_wait = (P.start != nullptr || P.rot_w > 0) ? 1 : 0;
    const int r = P.rope.rot_dim;
    const long long store_items = r / 16 + (kHeadDim - r) / 8 + kHeadDim / 8;
    const long long store_blocks =
        (static_cast<long long>(P.B) * P.T * store_items + kRopeThreads - 1) / kRopeThreads;
    const unsigned grid = static_cast<unsigned>(P.n_qtiles) * P.Hkv * P.B;
    cudaError_t err;
    if (P.start != nullptr) {
        // chunked prefill: store the chunk's keys and values first, clear the
        // never-written slots the last key tile may read, then attend over
        // the cache
        err = launch_overlapped(prefill_store_kv_kernel, dim3(static_cast<unsigned>(store_blocks)),
                                dim3(kRopeThreads), 0, stream, P);
        if (err != cudaSuccess) return err;
        err = launch_overlapped(cache_zero_tail_kernel, dim3(P.B), dim3(kRopeThreads), 0, stream,
                                P);
        if (err != cudaSuccess) return err;
        auto kernel = P.kind == kLayerSliding
                          ? attn_kernel_for<kKvFromRing, kLayerSliding>(P.G)
                          : attn_kernel_for<kKvFromCache, kLayerFull>(P.G);
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kAttnSmemBytes);
        if (err != cudaSuccess) return err;
        return launch_overlapped(kernel, dim3(grid), dim3(kAttnThreads), kAttnSmemBytes, stream,
                                 tm_q, tm_kv_k, tm_kv_v, tm_krot, tm_out, P);
    }
    if (P.rot_w > 0) {
        const long long items = r / 16 + (P.rot_w - r) / 8;
        const long long threads = static_cast<long long>(P.B) * P.T * items;
        const long long blocks = (threads + kRopeThreads - 1) / kRopeThreads;
        err = launch_overlapped(prefill_rope_k_kernel, dim3(static_cast<unsigned>(blocks)),
                                dim3(kRopeThreads), 0, stream, P);
        if (err != cudaSuccess) return err;
    }
    auto kernel = P.kind == kLayerSliding ? attn_kernel_for<kKvFromQkv, kLayerSliding>(P.G)
                                          : attn_kernel_for<kKvFromQkv, kKindAny>(P.G);
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kAttnSmemBytes);
    if (err != cudaSuccess) return err;
    err = launch_overlapped(kernel, dim3(grid), dim3(kAttnThreads), kAttnSmemBytes, stream, tm_q,
                            tm_kv_k, tm_kv_v, tm_krot, tm_out, P);
    if (err != cudaSuccess || P.k_cache == nullptr) return err;
    // fill the decode cache (it reads only qkv and pos)
    return launch_overlapped(prefill_store_kv_kernel, dim3(static_cast<unsigned>(store_blocks)),
                             dim3(kRopeThreads), 0, stream, P);
}

}  // namespace spark
