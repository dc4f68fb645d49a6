// host_io.cu -- prefill from and to host memory.
//
// A caller whose inputs sit in host memory would otherwise copy the whole
// batch in, run the prefill and copy the whole output back, one after the
// other.  Here the batch goes through kStages device staging areas one piece
// at a time -- a sequence, or a chunk (host_chunk tokens) of a longer one:
// copy-ins of later pieces and copy-outs of earlier ones run on two copy
// streams of the library while the caller's stream computes piece q.  A whole
// sequence runs the prefill with B = 1; chunks run the chunked prefill over a
// device KV cache of the sequence, which sees the same keys.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "common.cuh"
#include "spark_attn.h"

namespace spark {

spark_status prefill_impl(const void *qkv, const float *gate, const int32_t *pos,
                          const spark_layer_desc *desc, int B, int T, int H, int Hkv, void *out,
                          void *k_cache, void *v_cache, int64_t cap, const int32_t *start,
                          void *workspace, size_t workspace_bytes, void *stream,
                          bool validate_only);

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_copy_mu;
cudaStream_t g_copy_in[kMaxDevices] = {}, g_copy_out[kMaxDevices] = {};

// The library's two copy streams of the current device, created on first use.
bool copy_streams(cudaStream_t *in, cudaStream_t *out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(g_copy_mu);
    if (!g_copy_in[dev]) {
        cudaStream_t a = nullptr, b = nullptr;
        if (cudaStreamCreateWithFlags(&a, cudaStreamNonBlocking) != cudaSuccess) return false;
        if (cudaStreamCreateWithFlags(&b, cudaStreamNonBlocking) != cudaSuccess) {
            cudaStreamDestroy(a);
            return false;
        }
        g_copy_in[dev] = a;
        g_copy_out[dev] = b;
    }
    *in = g_copy_in[dev];
    *out = g_copy_out[dev];
    return true;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Sequences longer than this go through in chunks of this many tokens: the
// chunked prefill over a device KV cache (its query tiles and, on full
// layers, its key tiles fall where the one-shot prefill puts them).  Timed
// on one GB300 (4B shapes, B=2, T=8192, chunks of 1024 / 2048 / 3072 / 4096
// tokens): full layers 1.54 / 1.52 / 1.53 / 1.63 ms per call, sliding layers
// 1.51 / 1.39 / 1.33 / 1.41 ms.  A sliding chunk costs about the same
// wherever it sits (its keys end at the window), so longer chunks pay there;
// a full layer's last chunks walk the whole prefix.
int host_chunk(const spark_layer_desc *d) {
    return d->kind == SPARK_LAYER_SLIDING ? 3072 : 2048;
}
constexpr int kStages = 4;        // staging areas: pieces in flight

__global__ void chunk_starts_kernel(int32_t *starts, int n, int chunk) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) starts[i] = i * chunk;
}

// Workspace: the core's workspace for one piece (B = 1, T = chunk), the
// chunk start table and the KV cache of one sequence (chunked only), then
// kStages staging areas, each holding one piece's qkv, gate logits, positions
// and output.
struct HostPlan {
    int chunk, nchunks;
    int64_t cap;                  // cache slots (chunked only)
    size_t core_bytes, starts, k_cache, v_cache, stage0, stage_bytes, qkv, gate, pos, out, bytes;
};

HostPlan plan_host(size_t core_bytes, int T, int H, int Hkv, const spark_layer_desc *desc) {
    HostPlan pl{};
    pl.chunk = T > host_chunk(desc) ? host_chunk(desc) : T;
    pl.nchunks = (T + pl.chunk - 1) / pl.chunk;
    pl.core_bytes = core_bytes;
    size_t off = align256(core_bytes);
    if (pl.nchunks > 1) {
        // full layer: every token of the sequence; sliding: a ring that holds
        // the window plus one chunk, in whole 128-slot tiles
        pl.cap = desc->kind == SPARK_LAYER_FULL
                     ? T
                     : (static_cast<int64_t>(desc->window) + pl.chunk - 1 + 127) / 128 * 128;
        pl.starts = off;
        off += align256(static_cast<size_t>(pl.nchunks) * 4);
        const size_t cache = static_cast<size_t>(Hkv) * pl.cap * kHeadDim * 2;
        pl.k_cache = off;
        off += align256(cache);
        pl.v_cache = off;
        off += align256(cache);
    }
    pl.stage0 = off;
    const size_t C = static_cast<size_t>(pl.chunk);
    pl.qkv = 0;
    pl.gate = pl.qkv + align256(C * (H + 2 * Hkv) * kHeadDim * 2);
    pl.pos = pl.gate + align256(C * H * 4);
    pl.out = pl.pos + align256(C * 4);
    pl.stage_bytes = pl.out + align256(C * H * kHeadDim * 2);
    pl.bytes = pl.stage0 + kStages * pl.stage_bytes;
    return pl;
}

}  // namespace
}  // namespace spark

using namespace spark;

extern "C" {

size_t spark_attn_prefill_host_workspace_size(int B, int T, int H, int Hkv,
                                              const spark_layer_desc *desc) {
    if (B < 0 || T < 0 || !desc) return 0;
    const int chunk = T > host_chunk(desc) ? host_chunk(desc) : T;
    const size_t core = spark_attn_prefill_workspace_size(1, chunk, H, Hkv, desc);
    if (core == 0) return 0;
    return plan_host(core, T, H, Hkv, desc).bytes;
}

spark_status spark_attn_prefill_host(const void *qkv_h, const float *gate_h, const int32_t *pos_h,
                                     const spark_layer_desc *desc, int B, int T, int H, int Hkv,
                                     void *out_h, void *workspace, size_t workspace_bytes,
                                     void *stream) {
    if (!desc) return SPARK_ERR_NULL;
    if (B < 0 || T < 0) return SPARK_ERR_SHAPE;
    const int chunk0 = T > host_chunk(desc) ? host_chunk(desc) : T;
    const size_t core = spark_attn_prefill_workspace_size(1, chunk0, H, Hkv, desc);
    if (core == 0) {
        const spark_status st = prefill_impl(nullptr, nullptr, nullptr, desc, 1, T, H, Hkv,
                                             nullptr, nullptr, nullptr, 0, nullptr, nullptr, 0,
                                             stream, true);
        return st != SPARK_OK ? st : SPARK_ERR_SHAPE;
    }
    if (B == 0 || T == 0) return SPARK_OK;
    if (static_cast<long long>(B) * T > 0x7fffffffLL) return SPARK_ERR_UNSUPPORTED;
    if (!qkv_h || !gate_h || !pos_h || !out_h || !workspace) return SPARK_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return SPARK_ERR_ALIGN;
    const HostPlan pl = plan_host(core, T, H, Hkv, desc);
    if (workspace_bytes < pl.bytes) return SPARK_ERR_WORKSPACE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const bool chunked = pl.nchunks > 1;
    void *kc = chunked ? ws + pl.k_cache : nullptr;
    void *vc = chunked ? ws + pl.v_cache : nullptr;
    const int32_t *starts = chunked ? reinterpret_cast<int32_t *>(ws + pl.starts) : nullptr;
    auto stage = [&](int i) { return ws + pl.stage0 + static_cast<size_t>(i) * pl.stage_bytes; };
    // one piece of the batch: sequence b, tokens [c * chunk, c * chunk + len)
    auto run_piece = [&](uint8_t *sg, int c, int len, bool validate) {
        return prefill_impl(sg + pl.qkv, reinterpret_cast<float *>(sg + pl.gate),
                            reinterpret_cast<int32_t *>(sg + pl.pos), desc, 1, len, H, Hkv,
                            sg + pl.out, kc, vc, chunked ? pl.cap : 0,
                            chunked ? starts + c : nullptr, ws, pl.core_bytes, stream, validate);
    };
    // every check of the per-piece prefill, before anything is enqueued
    spark_status st = run_piece(stage(0), 0, pl.chunk, true);
    if (st != SPARK_OK) return st;
    cudaStream_t in = nullptr, out = nullptr;
    if (!copy_streams(&in, &out)) return SPARK_ERR_CUDA;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);

    const size_t qkv_tok = static_cast<size_t>(H + 2 * Hkv) * kHeadDim * 2;
    const size_t gate_tok = static_cast<size_t>(H) * 4, pos_tok = 4;
    const size_t out_tok = static_cast<size_t>(H) * kHeadDim * 2;
    const int pieces = B * pl.nchunks;
    // events: start, then per piece inputs in / computed / output out
    std::vector<cudaEvent_t> ev(1 + 3 * static_cast<size_t>(pieces), nullptr);
    auto cleanup = [&]() {
        for (cudaEvent_t e : ev)
            if (e) cudaEventDestroy(e);  // released once pending work has passed it
    };
    for (cudaEvent_t &e : ev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
            cleanup();
            return SPARK_ERR_CUDA;
        }
    cudaEvent_t start = ev[0];
    auto in_ready = [&](int q) { return ev[1 + 3 * q]; };
    auto computed = [&](int q) { return ev[2 + 3 * q]; };
    auto out_done = [&](int q) { return ev[3 + 3 * q]; };
    const uint8_t *qh = static_cast<const uint8_t *>(qkv_h);
    const uint8_t *gh = reinterpret_cast<const uint8_t *>(gate_h);
    const uint8_t *ph = reinterpret_cast<const uint8_t *>(pos_h);
    uint8_t *oh = static_cast<uint8_t *>(out_h);

    bool ok = cudaEventRecord(start, s) == cudaSuccess &&
              cudaStreamWaitEvent(in, start, 0) == cudaSuccess &&
              cudaStreamWaitEvent(out, start, 0) == cudaSuccess;
    if (ok && chunked) {
        chunk_starts_kernel<<<(pl.nchunks + 127) / 128, 128, 0, s>>>(
            reinterpret_cast<int32_t *>(ws + pl.starts), pl.nchunks, pl.chunk);
        ok = cudaGetLastError() == cudaSuccess;
    }
    for (int q = 0; ok && q < pieces; ++q) {
        const int b = q / pl.nchunks, c = q % pl.nchunks;
        const int t0 = c * pl.chunk;
        const int len = (T - t0 < pl.chunk) ? T - t0 : pl.chunk;
        const size_t tok0 = static_cast<size_t>(b) * T + t0;  // first token of the piece
        uint8_t *sg = stage(q % kStages);
        // copy-in: the staging inputs are free once the piece that used them is computed
        if (q >= kStages) ok = cudaStreamWaitEvent(in, computed(q - kStages), 0) == cudaSuccess;
        ok = ok &&
             cudaMemcpyAsync(sg + pl.qkv, qh + tok0 * qkv_tok, len * qkv_tok,
                             cudaMemcpyHostToDevice, in) == cudaSuccess &&
             cudaMemcpyAsync(sg + pl.gate, gh + tok0 * gate_tok, len * gate_tok,
                             cudaMemcpyHostToDevice, in) == cudaSuccess &&
             cudaMemcpyAsync(sg + pl.pos, ph + tok0 * pos_tok, len * pos_tok,
                             cudaMemcpyHostToDevice, in) == cudaSuccess &&
             cudaEventRecord(in_ready(q), in) == cudaSuccess;
        // compute: the staging output is free once its previous piece is copied out
        ok = ok && cudaStreamWaitEvent(s, in_ready(q), 0) == cudaSuccess;
        if (ok && q >= kStages)
            ok = cudaStreamWaitEvent(s, out_done(q - kStages), 0) == cudaSuccess;
        if (ok) {
            st = run_piece(sg, c, len, false);
            ok = st == SPARK_OK;
        }
        ok = ok && cudaEventRecord(computed(q), s) == cudaSuccess;
        // copy-out
        ok = ok && cudaStreamWaitEvent(out, computed(q), 0) == cudaSuccess &&
             cudaMemcpyAsync(oh + tok0 * out_tok, sg + pl.out, len * out_tok,
                             cudaMemcpyDeviceToHost, out) == cudaSuccess &&
             cudaEventRecord(out_done(q), out) == cudaSuccess;
    }
    // work ordered after this call on `stream` sees every output in host memory
    ok = ok && cudaStreamWaitEvent(s, out_done(pieces - 1), 0) == cudaSuccess;
    cleanup();
    if (!ok) return st != SPARK_OK ? st : SPARK_ERR_CUDA;
    return SPARK_OK;
}

}  // extern "C"
