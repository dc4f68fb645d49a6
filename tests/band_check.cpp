// Exhaustive CPU checks of the kernels' integer band logic (bands.cuh)
// against the mask definition of the Spark-X2.5 architecture page, §2:
// full layers are causal; a sliding layer's query i sees key j iff
// 0 <= i - j < window.  Built and driven by test_bands.py.
#include <cstdio>

#include "bands.cuh"

namespace {

// The definition, written out independently of bands.cuh.
bool visible(int kind, int window, long long i, long long j) {
    if (j > i) return false;
    if (kind == spark::kLayerSliding && i - j >= window) return false;
    return true;
}

}  // namespace

extern "C" {

// Every query tile [t0, t_end) of every sequence length up to t_max (tiles of
// tq tokens; the last tile of a length T ends at T), at absolute offset
// `start`: the visited key tiles cover every visible key, and neither the
// first nor the last tile is wholly invisible.  Returns the failures.
long long check_key_tiles(int kind, int window, int tq, int t_max, int start, int aligned) {
    const int tile = 128;
    long long bad = 0;
    for (int t0 = 0; t0 < t_max; t0 += tq) {
        for (int t_end = t0 + 1; t_end <= t0 + tq && t_end <= t_max; ++t_end) {
            const int a0 = start + t0, a_end = start + t_end;
            const spark::KeyTiles kt =
                spark::prefill_key_tiles(kind, window, a0, a_end, tile, aligned != 0);
            // first and last keys any query of the tile sees
            long long lo = a0;
            while (lo > 0 && visible(kind, window, a0, lo - 1)) --lo;
            const long long hi = a_end - 1;
            const long long tiles_end = static_cast<long long>(kt.kv_lo) + 128LL * kt.ntiles;
            bool ok = kt.ntiles >= 1 && kt.kv_lo >= 0 && kt.kv_lo <= lo && tiles_end > hi;
            ok = ok && lo < kt.kv_lo + tile;                              // first tile useful
            ok = ok && kt.kv_lo + static_cast<long long>(tile) * (kt.ntiles - 1) <= hi;
            if (aligned) ok = ok && kt.kv_lo % tile == 0;
            if (!ok) {
                if (bad < 3)
                    std::printf("key tiles: kind %d W %d tq %d start %d t0 %d t_end %d -> %d %d\n",
                                kind, window, tq, start, t0, t_end, kt.kv_lo, kt.ntiles);
                ++bad;
            }
        }
    }
    return bad;
}

// For every query tile up to t_max and every key tile it visits: a tile left
// unmasked is wholly visible from every query of the tile, and a tile that is
// wholly visible is left unmasked; key_visible matches the definition on
// every pair.  Returns the failures.
long long check_tile_masks(int kind, int window, int tq, int t_max, int start, int aligned) {
    const int tile = 128;
    long long bad = 0;
    for (int t0 = 0; t0 < t_max; t0 += tq) {
        const int t_end = (t0 + tq < t_max) ? t0 + tq : t_max;
        const int a0 = start + t0, a_last = start + t_end - 1;
        const spark::KeyTiles kt =
            spark::prefill_key_tiles(kind, window, a0, a_last + 1, tile, aligned != 0);
        for (int j = 0; j < kt.ntiles; ++j) {
            const int key0 = kt.kv_lo + j * tile;
            bool all = true, any = false;
            for (int q = a0; q <= a_last; ++q) {
                for (int k = key0; k < key0 + tile; ++k) {
                    const bool v = visible(kind, window, q, k);
                    if (v != spark::key_visible(kind, window, q, k)) ++bad;
                    all = all && v;
                    any = any || v;
                }
            }
            const bool need = spark::tile_needs_mask(kind, window, key0, tile, a0, a_last);
            if (need == all || !any) {
                if (bad < 3)
                    std::printf("mask: kind %d W %d tq %d start %d t0 %d tile %d need %d all %d any %d\n",
                                kind, window, tq, start, t0, j, need, all, any);
                ++bad;
            }
        }
    }
    return bad;
}

// Decode over a ring of `cap` slots (cap >= window): for every new-token
// position up to pos_max, the scanned slots are the filled ones and a slot is
// visible exactly when the token it holds is inside the window.  The
// visible slots plus the new token are exactly the window's tokens.
long long check_ring(int cap, int window, long long pos_max) {
    long long bad = 0;
    for (long long pos = 0; pos <= pos_max; ++pos) {
        const long long n = spark::decode_scan_slots(spark::kLayerSliding, pos, cap);
        if (n != (pos < cap ? pos : cap)) ++bad;
        long long seen = 0;
        for (long long s = 0; s < n; ++s) {
            long long j = -1;  // the latest token j < pos written to slot s
            for (long long t = pos - 1; t >= 0 && t >= pos - cap; --t)
                if (t % cap == s) { j = t; break; }
            const bool want = j >= 0 && visible(spark::kLayerSliding, window, pos, j);
            const bool got = spark::ring_slot_visible(s, pos, cap, window);
            if (want != got) {
                if (bad < 3)
                    std::printf("ring: cap %d W %d pos %lld slot %lld want %d got %d\n", cap,
                                window, pos, s, want, got);
                ++bad;
            }
            seen += got;
        }
        const long long window_tokens = (pos + 1 < window ? pos + 1 : window);
        if (seen + 1 != window_tokens) ++bad;
        if (spark::decode_scan_slots(spark::kLayerFull, pos, cap) != pos) ++bad;
    }
    return bad;
}

}  // extern "C"
