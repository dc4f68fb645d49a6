// bands.cuh -- the integer band logic of the attention core: which keys a
// query sees, which key tiles a query tile visits and which of those need a
// per-element mask, and which cache slots a decode step sees.  The kernels
// and the CPU tests compile this same header, so the tests check exactly what
// the kernels run.
//
// Spark-X2.5 architecture (4B / 1.7B), §2: full_attention layers are causal;
// sliding_attention layers see the latest `window` tokens, the query
// included (key j visible from query i iff 0 <= i - j < window).
// Spark-X2.5-4B hybrid-attention explainer (lshu.cn): a sliding layer's cache
// keeps only the latest tokens, so decode reads a ring of slots.
#pragma once

#if defined(__CUDACC__)
#define SPARK_HD __host__ __device__ __forceinline__
#else
#define SPARK_HD inline
#endif

namespace spark {

constexpr int kLayerFull = 0;
constexpr int kLayerSliding = 1;

// Key `key` is visible from query `q` (absolute token indices of a prefill).
SPARK_HD bool key_visible(int kind, int window, int q, int key) {
    return key <= q && (kind == kLayerFull || q - key < window);
}

struct KeyTiles {
    int kv_lo;   // first key of the first tile
    int ntiles;  // tiles of `tile` keys from kv_lo
};

// Key tiles that the queries [a0, a_end) (a_end > a0) visit: from the first key
// any of them sees to the last query.  With `aligned`, kv_lo is rounded down
// to a multiple of `tile` (a power of two), as reads from a ring need.
SPARK_HD KeyTiles prefill_key_tiles(int kind, int window, int a0, int a_end, int tile,
                                    bool aligned) {
    int lo = (kind == kLayerFull) ? 0 : (a0 - window + 1 > 0 ? a0 - window + 1 : 0);
    if (aligned) lo &= ~(tile - 1);
    return KeyTiles{lo, (a_end - lo + tile - 1) / tile};
}

// Whether the keys [key0, key0 + tile) need a per-element mask for the queries
// [a0, a_last]: false only when every one of them is visible from every query.
SPARK_HD bool tile_needs_mask(int kind, int window, int key0, int tile, int a0, int a_last) {
    return (key0 + tile - 1 > a0) || (kind == kLayerSliding && a_last - key0 >= window);
}

// Decode: the cache slots [0, n) scanned before the new token at `pos` is
// merged in (every past token of a full layer; the filled part of a ring).
SPARK_HD long long decode_scan_slots(int kind, long long pos, long long cap) {
    return (kind == kLayerFull) ? pos : (pos < cap ? pos : cap);
}

// Slot s (s < min(pos, cap)) of a ring of `cap` slots holds the latest token
// j < pos with j = s (mod cap).  It is visible from the new token at `pos`
// iff pos - j < window.
SPARK_HD bool ring_slot_visible(long long s, long long pos, long long cap, int window) {
    const long long j = s + cap * ((pos - 1 - s) / cap);
    return pos - j < static_cast<long long>(window);
}

}  // namespace spark
