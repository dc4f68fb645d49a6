// c_abi_example.cpp -- the library driven from C++ alone, without Python.
//
// A sliding-layer prefill that fills a 512-slot ring (spark_attn_prefill_cache),
// then one decode step over that ring (spark_attn_decode), on device buffers
// this program allocates itself, with the status word read back at the end.
// It also makes one call with an invalid head count, which must be refused on
// the host.  Inputs are read from files the test writes; the outputs are
// written next to them for the test to compare with the Python binding's.
//
//   c_abi_example <dir> <B> <T> <H> <Hkv>
//   in:  qkv.bin bf16 [B,T,(H+2Hkv)*256], gate.bin f32 [B,T,H], pos.bin i32 [B,T],
//        qkv1.bin bf16 [B,(H+2Hkv)*256], gate1.bin f32 [B,H], pos1.bin i32 [B]
//   out: out.bin bf16 [B,T,H*256], y.bin bf16 [B,H*256]
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <string>
#include <vector>

#include "spark_attn.h"

namespace {

std::vector<char> read_file(const std::string &path, size_t bytes) {
    std::vector<char> buf(bytes);
    FILE *f = std::fopen(path.c_str(), "rb");
    if (!f || std::fread(buf.data(), 1, bytes, f) != bytes) {
        std::fprintf(stderr, "cannot read %zu bytes from %s\n", bytes, path.c_str());
        std::exit(2);
    }
    std::fclose(f);
    return buf;
}

void write_file(const std::string &path, const void *data, size_t bytes) {
    FILE *f = std::fopen(path.c_str(), "wb");
    if (!f || std::fwrite(data, 1, bytes, f) != bytes) {
        std::fprintf(stderr, "cannot write %s\n", path.c_str());
        std::exit(2);
    }
    std::fclose(f);
}

void *to_device(const std::vector<char> &host) {
    void *p = nullptr;
    if (cudaMalloc(&p, host.size()) != cudaSuccess ||
        cudaMemcpy(p, host.data(), host.size(), cudaMemcpyHostToDevice) != cudaSuccess) {
        std::fprintf(stderr, "device copy failed\n");
        std::exit(3);
    }
    return p;
}

void check(spark_status st, const char *what) {
    if (st != SPARK_OK) {
        std::fprintf(stderr, "%s: %s\n", what, spark_status_str(st));
        std::exit(4);
    }
}

}  // namespace

int main(int argc, char **argv) {
    if (argc != 6) {
        std::fprintf(stderr, "usage: %s dir B T H Hkv\n", argv[0]);
        return 1;
    }
    const std::string dir = argv[1];
    const int B = std::atoi(argv[2]), T = std::atoi(argv[3]);
    const int H = std::atoi(argv[4]), Hkv = std::atoi(argv[5]);
    const size_t width = static_cast<size_t>(H + 2 * Hkv) * SPARK_HEAD_DIM;
    const int64_t cap = 512;
    const spark_layer_desc sliding = {SPARK_LAYER_SLIDING, 512, 1e4, 256, SPARK_GATE_SIGMOID};

    void *qkv = to_device(read_file(dir + "/qkv.bin", size_t(B) * T * width * 2));
    void *gate = to_device(read_file(dir + "/gate.bin", size_t(B) * T * H * 4));
    void *pos = to_device(read_file(dir + "/pos.bin", size_t(B) * T * 4));
    void *qkv1 = to_device(read_file(dir + "/qkv1.bin", size_t(B) * width * 2));
    void *gate1 = to_device(read_file(dir + "/gate1.bin", size_t(B) * H * 4));
    void *pos1 = to_device(read_file(dir + "/pos1.bin", size_t(B) * 4));

    const size_t out_bytes = size_t(B) * T * H * SPARK_HEAD_DIM * 2;
    const size_t y_bytes = size_t(B) * H * SPARK_HEAD_DIM * 2;
    const size_t cache_bytes = size_t(B) * Hkv * cap * SPARK_HEAD_DIM * 2;
    size_t ws_bytes = spark_attn_prefill_workspace_size(B, T, H, Hkv, &sliding);
    const size_t dec_ws = spark_attn_decode_workspace_size(B, H, Hkv, cap, &sliding);
    if (ws_bytes == 0 || dec_ws == 0) check(SPARK_ERR_SHAPE, "workspace size query");
    if (dec_ws > ws_bytes) ws_bytes = dec_ws;
    void *out = nullptr, *y = nullptr, *kc = nullptr, *vc = nullptr, *ws = nullptr;
    if (cudaMalloc(&out, out_bytes) != cudaSuccess || cudaMalloc(&y, y_bytes) != cudaSuccess ||
        cudaMalloc(&kc, cache_bytes) != cudaSuccess || cudaMalloc(&vc, cache_bytes) != cudaSuccess ||
        cudaMalloc(&ws, ws_bytes) != cudaSuccess || cudaMemset(ws, 0, ws_bytes) != cudaSuccess) {
        std::fprintf(stderr, "allocation failed\n");
        return 3;
    }
    cudaStream_t stream = nullptr;
    if (cudaStreamCreate(&stream) != cudaSuccess) return 3;

    // a head count that does not divide the query heads is refused before any work
    const spark_status bad = spark_attn_prefill(qkv, static_cast<const float *>(gate),
                                                static_cast<const int32_t *>(pos), &sliding, B,
                                                T, H, 3, out, ws, ws_bytes, stream);
    if (bad == SPARK_OK) {
        std::fprintf(stderr, "an invalid head count was accepted\n");
        return 5;
    }

    check(spark_attn_prefill_cache(qkv, static_cast<const float *>(gate),
                                   static_cast<const int32_t *>(pos), kc, vc, cap, &sliding, B, T,
                                   H, Hkv, out, ws, ws_bytes, stream),
          "spark_attn_prefill_cache");
    check(spark_attn_decode(qkv1, static_cast<const float *>(gate1),
                            static_cast<const int32_t *>(pos1), kc, vc, cap, &sliding, B, H, Hkv,
                            y, ws, ws_bytes, stream),
          "spark_attn_decode");
    uint32_t device_status = 0xffffffffu;
    check(spark_attn_read_status(ws, &device_status, 0, stream), "spark_attn_read_status");

    std::vector<char> out_h(out_bytes), y_h(y_bytes);
    if (cudaMemcpy(out_h.data(), out, out_bytes, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(y_h.data(), y, y_bytes, cudaMemcpyDeviceToHost) != cudaSuccess)
        return 3;
    write_file(dir + "/out.bin", out_h.data(), out_bytes);
    write_file(dir + "/y.bin", y_h.data(), y_bytes);
    std::printf("ok status=%u refused=%s version=%s\n", device_status, spark_status_str(bad),
                spark_attn_version());
    return device_status == 0 ? 0 : 6;
}
