// host_io.cu -- prefill from and to host memory.
//
// A caller whose inputs sit in host memory would otherwise copy the whole
// batch in, run the prefill and copy the whole output back, one after the
// other.  Here the batch goes through two device staging areas one sequence
// at a time: the copy-in of sequence b+1 and the copy-out of sequence b-1 run
// on two copy streams of the library while the caller's stream computes
// sequence b (the same prefill, with B = 1).
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

// Workspace: the core's workspace for one sequence, then two staging areas,
// each holding one sequence's qkv, gate logits, positions and output.
struct HostPlan {
    size_t core_bytes, stage0, stage_bytes, qkv, gate, pos, out, bytes;
};

HostPlan plan_host(size_t core_bytes, int T, int H, int Hkv) {
    HostPlan pl{};
    pl.core_bytes = core_bytes;
    pl.stage0 = align256(core_bytes);
    pl.qkv = 0;
    pl.gate = pl.qkv + align256(static_cast<size_t>(T) * (H + 2 * Hkv) * kHeadDim * 2);
    pl.pos = pl.gate + align256(static_cast<size_t>(T) * H * 4);
    pl.out = pl.pos + align256(static_cast<size_t>(T) * 4);
    pl.stage_bytes = pl.out + align256(static_cast<size_t>(T) * H * kHeadDim * 2);
    pl.bytes = pl.stage0 + 2 * pl.stage_bytes;
    return pl;
}

}  // namespace
}  // namespace spark

using namespace spark;

extern "C" {

size_t spark_attn_prefill_host_workspace_size(int B, int T, int H, int Hkv,
                                              const spark_layer_desc *desc) {
    if (B < 0 || T < 0) return 0;
    const size_t core = spark_attn_prefill_workspace_size(1, T, H, Hkv, desc);
    if (core == 0) return 0;
    return plan_host(core, T, H, Hkv).bytes;
}

spark_status spark_attn_prefill_host(const void *qkv_h, const float *gate_h, const int32_t *pos_h,
                                     const spark_layer_desc *desc, int B, int T, int H, int Hkv,
                                     void *out_h, void *workspace, size_t workspace_bytes,
                                     void *stream) {
    if (!desc) return SPARK_ERR_NULL;
    if (B < 0 || T < 0) return SPARK_ERR_SHAPE;
    const size_t core = spark_attn_prefill_workspace_size(1, T, H, Hkv, desc);
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
    const HostPlan pl = plan_host(core, T, H, Hkv);
    if (workspace_bytes < pl.bytes) return SPARK_ERR_WORKSPACE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    auto stage = [&](int i) { return ws + pl.stage0 + static_cast<size_t>(i) * pl.stage_bytes; };
    // every check of the per-sequence prefill, before anything is enqueued
    spark_status st = prefill_impl(stage(0) + pl.qkv, reinterpret_cast<float *>(stage(0) + pl.gate),
                                   reinterpret_cast<int32_t *>(stage(0) + pl.pos), desc, 1, T, H,
                                   Hkv, stage(0) + pl.out, nullptr, nullptr, 0, nullptr, ws,
                                   pl.core_bytes, stream, true);
    if (st != SPARK_OK) return st;
    cudaStream_t in = nullptr, out = nullptr;
    if (!copy_streams(&in, &out)) return SPARK_ERR_CUDA;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);

    const size_t qkv_seq = static_cast<size_t>(T) * (H + 2 * Hkv) * kHeadDim * 2;
    const size_t gate_seq = static_cast<size_t>(T) * H * 4, pos_seq = static_cast<size_t>(T) * 4;
    const size_t out_seq = static_cast<size_t>(T) * H * kHeadDim * 2;
    // events: start, then per sequence inputs in / computed / output out
    std::vector<cudaEvent_t> ev(1 + 3 * static_cast<size_t>(B), nullptr);
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
    auto in_ready = [&](int b) { return ev[1 + 3 * b]; };
    auto computed = [&](int b) { return ev[2 + 3 * b]; };
    auto out_done = [&](int b) { return ev[3 + 3 * b]; };
    const uint8_t *qh = static_cast<const uint8_t *>(qkv_h);
    const uint8_t *gh = reinterpret_cast<const uint8_t *>(gate_h);
    const uint8_t *ph = reinterpret_cast<const uint8_t *>(pos_h);
    uint8_t *oh = static_cast<uint8_t *>(out_h);

    bool ok = cudaEventRecord(start, s) == cudaSuccess &&
              cudaStreamWaitEvent(in, start, 0) == cudaSuccess &&
              cudaStreamWaitEvent(out, start, 0) == cudaSuccess;
    for (int b = 0; ok && b < B; ++b) {
        uint8_t *sg = stage(b & 1);
        // copy-in: the staging inputs are free once sequence b-2 is computed
        if (b >= 2) ok = cudaStreamWaitEvent(in, computed(b - 2), 0) == cudaSuccess;
        ok = ok &&
             cudaMemcpyAsync(sg + pl.qkv, qh + b * qkv_seq, qkv_seq, cudaMemcpyHostToDevice, in) ==
                 cudaSuccess &&
             cudaMemcpyAsync(sg + pl.gate, gh + b * gate_seq, gate_seq, cudaMemcpyHostToDevice,
                             in) == cudaSuccess &&
             cudaMemcpyAsync(sg + pl.pos, ph + b * pos_seq, pos_seq, cudaMemcpyHostToDevice, in) ==
                 cudaSuccess &&
             cudaEventRecord(in_ready(b), in) == cudaSuccess;
        // compute: the staging output is free once sequence b-2 is copied out
        ok = ok && cudaStreamWaitEvent(s, in_ready(b), 0) == cudaSuccess;
        if (ok && b >= 2) ok = cudaStreamWaitEvent(s, out_done(b - 2), 0) == cudaSuccess;
        if (ok) {
            st = prefill_impl(sg + pl.qkv, reinterpret_cast<float *>(sg + pl.gate),
                              reinterpret_cast<int32_t *>(sg + pl.pos), desc, 1, T, H, Hkv,
                              sg + pl.out, nullptr, nullptr, 0, nullptr, ws, pl.core_bytes, stream,
                              false);
            ok = st == SPARK_OK;
        }
        ok = ok && cudaEventRecord(computed(b), s) == cudaSuccess;
        // copy-out
        ok = ok && cudaStreamWaitEvent(out, computed(b), 0) == cudaSuccess &&
             cudaMemcpyAsync(oh + b * out_seq, sg + pl.out, out_seq, cudaMemcpyDeviceToHost,
                             out) == cudaSuccess &&
             cudaEventRecord(out_done(b), out) == cudaSuccess;
    }
    // work ordered after this call on `stream` sees every output in host memory
    ok = ok && cudaStreamWaitEvent(s, out_done(B - 1), 0) == cudaSuccess;
    cleanup();
    if (!ok) return st != SPARK_OK ? st : SPARK_ERR_CUDA;
    return SPARK_OK;
}

}  // extern "C"
