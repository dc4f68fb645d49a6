// gemm.cu -- the dense projections of the attention block on the 5th-generation
// tensor cores: y = x W^T in bf16 with fp32 accumulation in TMEM.
//
// Spark-X2.5 architecture (4B / 1.7B), §3 Eq. 1 and Fig. 1: q_k_v_proj
// (hidden -> (H + 2 Hkv) * 256) and g_proj (hidden -> H) read the normed
// hidden state, out_proj (H * 256 -> hidden) maps the gated attention output
// back; §6 gives the 4B sizes 2560 -> 6144, 2560 -> 16 and 4096 -> 2560.
// Weights use the PyTorch Linear layout W [N, K] (row major), so both
// operands are K-major.  Every product is rounded once to bf16, the
// checkpoints' dtype (§1).
//
// One persistent kernel, one CTA per SM, walking output tiles of 128 rows x
// 256 columns with the columns fastest, so that the CTAs running at once
// share a few row blocks of x and all of W in L2.  An optional second weight
// W2 [N2, K] (g_proj, N2 <= 256) adds one tile column of N2 rounded up to 16
// per row block: its products go to a second output as fp32 values that hold
// the bf16-rounded result, so the gate logits leave the kernel already in the
// Linear's output dtype.
//
// With rope_heads > 0 (q_k_v_proj of the attention block) the epilogue also
// applies RoPE (§4 layered RoPE; rotate_half pairs (k, k + r/2) of the first r
// dims, angle pos * theta^(-2k/r)) to the first rope_heads output heads, the
// H query heads and Hkv key heads: a 256-column tile is exactly one head.  It
// rounds the fp32 product to bf16 first (the Linear's output), then rotates in
// fp32 and rounds again, the order and arithmetic of the attention core's own
// rotation, so the core can run on the result without rotating.
//
// Warp roles:
//   warp 0       TMA producer: per k-step of 64, the x tile (128 x 64) and the
//                W tile (256 x 64, or N2 rounded up x 64), 128-byte swizzle,
//                into a ring of kGemmStages stages
//   warp 1       TMEM owner (512 columns: two 128 x 256 fp32 accumulators)
//                and MMA issuer (one thread): M128 N256 K16 products
//   warps 4..11  epilogue, two warpgroups: output row i is TMEM lane i;
//                warpgroup w converts columns [128w, 128w + 128) of a finished
//                tile and stores them while the MMA thread fills the other
//                accumulator with the CTA's next tile
// Every wait is bounded (ptx.cuh): a wait that gives up sets kErrTimeout in
// the status word and the CTA drains its copies and products and returns.
#include <cudaTypedefs.h>

#include <climits>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "spark_attn.h"

namespace spark {

constexpr int kGemmBM = 128;
constexpr int kGemmBN = 256;
constexpr int kGemmBK = 64;                                    // one 128-byte swizzle row
constexpr int kGemmStages = 4;
constexpr int kGemmABytes = kGemmBM * kGemmBK * 2;             // 16 KB
constexpr int kGemmBBytes = kGemmBN * kGemmBK * 2;             // 32 KB
constexpr int kGemmThreads = 384;
constexpr int kGemmEpiWarp0 = 4;
constexpr int kGemmEpiThreads = 256;
constexpr uint32_t kGemmTmemCols = 512;

// barriers
constexpr int kGBarFull = 0;                        // kGemmStages
constexpr int kGBarEmpty = kGemmStages;             // kGemmStages
constexpr int kGBarAccFull = 2 * kGemmStages;       // 2
constexpr int kGBarAccEmpty = 2 * kGemmStages + 2;  // 2 (one arrival per epilogue warp)
constexpr int kGBarDrain = 2 * kGemmStages + 4;
constexpr int kGNumBars = 2 * kGemmStages + 5;

constexpr int kGemmSmemBytes = 1024 + kGemmStages * (kGemmABytes + kGemmBBytes) + 256;

struct GemmParams {
    void *out;          // [M, N] bf16 (row stride ldo elements)
    float *out2;        // [M, N2] fp32 holding bf16-rounded values (when N2 > 0)
    unsigned *status;   // device status word (kErrTimeout)
    const int32_t *pos; // [M] positions of the rows (rope_heads > 0)
    int M, N, K;
    int ldo;
    int N2;             // rows of W2 (0: none)
    int m_tiles, n_tiles;  // tiles of the main product
    int rope_heads;     // leading 256-column tiles rotated in the epilogue (0: none);
                        // rope.rot_dim / 2 is then a multiple of 32
    RopeTable rope;
};

// Rounds an fp32 product to bf16 and back (the Linear's bf16 output).
__device__ __forceinline__ float round_bf16(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}

// Stores 32 consecutive bf16 outputs from packed pairs (masked to N).
__device__ __forceinline__ void store32(__nv_bfloat16 *dst, const uint32_t (&pk)[16], int n0,
                                        int N) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (n0 + 8 * q + 8 > N) break;
        *reinterpret_cast<uint4 *>(dst + 8 * q) =
            make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tm_x,
                     const __grid_constant__ CUtensorMap tm_w,
                     const __grid_constant__ CUtensorMap tm_w2,
                     const __grid_constant__ GemmParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *abuf = smem;                                   // kGemmStages x 16 KB
    uint8_t *bbuf = smem + kGemmStages * kGemmABytes;       // kGemmStages x 32 KB
    uint64_t *bars = reinterpret_cast<uint64_t *>(bbuf + kGemmStages * kGemmBBytes);
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int col_tiles = P.n_tiles + (P.N2 > 0 ? 1 : 0);
    const int total = P.m_tiles * col_tiles;
    const int ksteps = (P.K + kGemmBK - 1) / kGemmBK;
    const int n2_pad = (P.N2 + 15) / 16 * 16;
    const uint32_t b2_bytes = static_cast<uint32_t>(n2_pad) * kGemmBK * 2;

    if (tid == 0) {
        for (int i = 0; i < kGNumBars; ++i) {
            const bool acc_empty = i == kGBarAccEmpty || i == kGBarAccEmpty + 1;
            mbar_init(&bars[i], acc_empty ? kGemmEpiThreads / 32 : 1);
        }
        fence_mbar_init();
        abort_flag = 0;
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base_sh, kGemmTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
        if (P.N2 > 0) tma_prefetch_desc(&tm_w2);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    // x may be the previous kernel's output, and the outputs may still be
    // read by it (programmatic dependent launch)
    grid_dep_wait();
    grid_dep_launch();

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        int sc = 0;  // stages filled so far
        if (lane == 0) {
            bool ok = true;
            for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
                const int mt = t / col_tiles, nt = t % col_tiles;
                const bool second = nt == P.n_tiles;
                for (int k = 0; k < ksteps; ++k) {
                    const int s = sc % kGemmStages;
                    if (sc >= kGemmStages &&
                        !mbar_wait(&bars[kGBarEmpty + s], ((sc / kGemmStages) - 1) & 1,
                                   &abort_flag, P.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars[kGBarFull + s],
                                          kGemmABytes + (second ? b2_bytes : kGemmBBytes));
                    tma_load_2d(abuf + s * kGemmABytes, &tm_x, &bars[kGBarFull + s], k * kGemmBK,
                                mt * kGemmBM);
                    if (second)
                        tma_load_2d(bbuf + s * kGemmBBytes, &tm_w2, &bars[kGBarFull + s],
                                    k * kGemmBK, 0);
                    else
                        tma_load_2d(bbuf + s * kGemmBBytes, &tm_w, &bars[kGBarFull + s],
                                    k * kGemmBK, nt * kGemmBN);
                    ++sc;
                }
            }
        }
        __syncwarp();
        tc_fence_before();
        __syncthreads();
        // after an abort, copies in flight must land before shared memory is released
        if (lane == 0 && abort_flag) {
            const int first = sc > kGemmStages ? sc - kGemmStages : 0;
            for (int s = first; s < sc; ++s)
                mbar_wait_plain(&bars[kGBarFull + (s % kGemmStages)], (s / kGemmStages) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            // descriptors built once; an operand at byte offset o from a base
            // has the base's descriptor plus o / 16 (every address < 2^18)
            const uint64_t a_desc = smem_desc_sw128(smem_u32(abuf), 16, 1024);
            const uint64_t b_desc = smem_desc_sw128(smem_u32(bbuf), 16, 1024);
            const uint32_t idesc_main = idesc_bf16_f32(kGemmBM, kGemmBN, 0, 0);
            const uint32_t idesc_second = idesc_bf16_f32(kGemmBM, n2_pad > 0 ? n2_pad : 16, 0, 0);
            int sc = 0;
            bool ok = true;
            int it = 0;
            for (int t = blockIdx.x; ok && t < total; t += gridDim.x, ++it) {
                const bool second = (t % col_tiles) == P.n_tiles;
                const int buf = it & 1;
                if (it >= 2 && !mbar_wait(&bars[kGBarAccEmpty + buf], ((it >> 1) - 1) & 1,
                                          &abort_flag, P.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(buf * kGemmBN);
                const uint32_t idesc = second ? idesc_second : idesc_main;
                for (int k = 0; k < ksteps; ++k) {
                    const int s = sc % kGemmStages;
                    if (!mbar_wait(&bars[kGBarFull + s], (sc / kGemmStages) & 1, &abort_flag,
                                   P.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kGemmBK / 16; ++kk) {
                        const uint64_t ad =
                            a_desc + static_cast<uint32_t>((s * kGemmABytes + kk * 32) >> 4);
                        const uint64_t bd =
                            b_desc + static_cast<uint32_t>((s * kGemmBBytes + kk * 32) >> 4);
                        mma_ss(d, ad, bd, idesc, (k | kk) != 0);
                    }
                    tc_commit(&bars[kGBarEmpty + s]);
                    ++sc;
                }
                if (ok) tc_commit(&bars[kGBarAccFull + buf]);
            }
            // every product issued so far must finish before TMEM is released
            tc_commit(&bars[kGBarDrain]);
            mbar_wait_plain(&bars[kGBarDrain], 0);
        }
        __syncwarp();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        tmem_dealloc(tmem, kGemmTmemCols);
    } else if (warp >= kGemmEpiWarp0) {
        // ------------------------------------------------------ epilogue
        const int wq = warp & 3;                        // TMEM lane quarter
        const int wg = (warp - kGemmEpiWarp0) >> 2;     // column half
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(P.out);
        int it = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
            const int mt = t / col_tiles, nt = t % col_tiles;
            const bool second = nt == P.n_tiles;
            const int buf = it & 1;
            if (!mbar_wait(&bars[kGBarAccFull + buf], (it >> 1) & 1, &abort_flag, P.status))
                break;
            tc_fence_after();
            const int row = mt * kGemmBM + wq * 32 + lane;
            const uint32_t acc = lane_base + static_cast<uint32_t>(buf * kGemmBN);
            if (!second && nt >= P.rope_heads) {
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    const int col = wg * 128 + c * 32;
                    uint32_t v[32];
                    tmem_ld32(acc + col, v);
                    tmem_ld_wait();
                    const int n0 = nt * kGemmBN + col;
                    if (row < P.M) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]),
                                                __uint_as_float(v[2 * i + 1]));
                        store32(out + static_cast<size_t>(row) * P.ldo + n0, pk, n0, P.N);
                    }
                }
            } else if (!second) {
                // a query or key head: pairs (k, k + r/2) for k < r/2, in units
                // of 32 pairs (two 32-column chunks), then the unrotated
                // chunks; the two warpgroups take alternate units
                const int r = P.rope.rot_dim, half = r / 2;
                const int npair = half / 32, nunits = npair + (kGemmBN - r) / 32;
                const int p = row < P.M ? P.pos[row] : 0;
                __nv_bfloat16 *dst = out + static_cast<size_t>(row < P.M ? row : 0) * P.ldo +
                                     nt * kGemmBN;
#pragma unroll 1
                for (int u = wg; u < nunits; u += 2) {
                    if (u < npair) {
                        const int c1 = u * 32, c2 = c1 + half;
                        uint32_t v1[32], v2[32];
                        tmem_ld32(acc + c1, v1);
                        tmem_ld32(acc + c2, v2);
                        tmem_ld_wait();
                        uint32_t pa[16], pb[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float y[2][2];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                float cs, sn;
                                rope_cos_sin(p, P.rope.u[c1 + 2 * i + e], cs, sn);
                                rope_rotate(round_bf16(__uint_as_float(v1[2 * i + e])),
                                            round_bf16(__uint_as_float(v2[2 * i + e])), cs, sn,
                                            y[0][e], y[1][e]);
                            }
                            pa[i] = pack_bf16x2(y[0][0], y[0][1]);
                            pb[i] = pack_bf16x2(y[1][0], y[1][1]);
                        }
                        if (row < P.M) {
                            store32(dst + c1, pa, nt * kGemmBN + c1, P.N);
                            store32(dst + c2, pb, nt * kGemmBN + c2, P.N);
                        }
                    } else {
                        const int c = r + (u - npair) * 32;
                        uint32_t v[32];
                        tmem_ld32(acc + c, v);
                        tmem_ld_wait();
                        if (row < P.M) {
                            uint32_t pk[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]),
                                                    __uint_as_float(v[2 * i + 1]));
                            store32(dst + c, pk, nt * kGemmBN + c, P.N);
                        }
                    }
                }
            } else if (wg == 0) {
                // the second product: N2 <= 256 columns, 32 at a time
                for (int col = 0; col < n2_pad; col += 32) {
                    uint32_t v[32];
                    tmem_ld32(acc + col, v);
                    tmem_ld_wait();
                    if (row < P.M) {
                        float *dst = P.out2 + static_cast<size_t>(row) * P.N2;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col + j < P.N2) dst[col + j] = round_bf16(__uint_as_float(v[j]));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kGBarAccEmpty + buf]);
        }
        tc_fence_before();
        __syncthreads();
    } else {
        // warps 2 and 3 have no role
        __syncthreads();
    }
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 gemm_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        cudaGetLastError();
    });
    return fn;
}

// A row-major bf16 matrix [rows, K] as a 2-D tensor map with boxes of
// box_rows x 64, 128-byte swizzle.
bool encode_rows(CUtensorMap *map, const void *base, long long rows, int K, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = gemm_encode_fn();
    if (!fn) return false;
    cuuint64_t gd[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    cuuint64_t gs[1] = {static_cast<cuuint64_t>(K) * 2};
    cuuint32_t bx[2] = {static_cast<cuuint32_t>(kGemmBK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t es[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), gd, gs, bx, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

int gemm_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 152;
    }
    return sms;
}

}  // namespace

// The checks of launch_linear, without a launch: SPARK_OK or the status the
// call would return.
spark_status check_linear(const void *x, const void *w, void *y, long long M, int N, int K,
                          const void *w2, float *y2, int N2) {
    if (M < 0 || N <= 0 || K <= 0 || N2 < 0) return SPARK_ERR_SHAPE;
    if (M > 0x7fffffffLL - kGemmBM) return SPARK_ERR_UNSUPPORTED;
    if (N % 8 != 0 || K % 8 != 0 || N2 > kGemmBN) return SPARK_ERR_UNSUPPORTED;
    const long long tiles = (M + kGemmBM - 1) / kGemmBM * ((N + kGemmBN - 1) / kGemmBN + 1);
    if (tiles > INT_MAX) return SPARK_ERR_UNSUPPORTED;
    if (M == 0) return SPARK_OK;
    if (!x || !w || !y || (N2 > 0 && (!w2 || !y2))) return SPARK_ERR_NULL;
    auto al = [](const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; };
    if (!al(x, 16) || !al(w, 16) || !al(y, 16) || (N2 > 0 && (!al(w2, 16) || !al(y2, 4))))
        return SPARK_ERR_ALIGN;
    return SPARK_OK;
}

// y[M, N] = bf16(x[M, K] W[N, K]^T), and with N2 > 0 also
// y2[M, N2] = float(bf16(x W2[N2, K]^T)).  status: device status word.  With
// rope != nullptr the first rope_heads 256-column heads of y are rotated at
// the positions pos[M] (rope->rot_dim / 2 a multiple of 32, N >= rope_heads * 256).
spark_status launch_linear(const void *x, const void *w, void *y, long long M, int N, int K,
                           const void *w2, float *y2, int N2, unsigned *status,
                           cudaStream_t stream, const RopeTable *rope, const int32_t *pos,
                           int rope_heads) {
    spark_status st = check_linear(x, w, y, M, N, K, w2, y2, N2);
    if (st != SPARK_OK || M == 0) return st;
    if (rope && rope_heads > 0 &&
        (!pos || (rope->rot_dim / 2) % 32 != 0 || static_cast<long long>(rope_heads) * kGemmBN > N))
        return SPARK_ERR_UNSUPPORTED;
    CUtensorMap tm_x, tm_w, tm_w2;
    std::memset(&tm_w2, 0, sizeof(tm_w2));
    if (!encode_rows(&tm_x, x, M, K, kGemmBM) || !encode_rows(&tm_w, w, N, K, kGemmBN))
        return SPARK_ERR_CUDA;
    if (N2 > 0 && !encode_rows(&tm_w2, w2, N2, K, (N2 + 15) / 16 * 16)) return SPARK_ERR_CUDA;
    GemmParams P;
    std::memset(&P, 0, sizeof(P));
    P.out = y;
    P.out2 = y2;
    P.status = status;
    P.M = static_cast<int>(M);
    P.N = N;
    P.K = K;
    P.ldo = N;
    P.N2 = N2;
    P.m_tiles = static_cast<int>((M + kGemmBM - 1) / kGemmBM);
    P.n_tiles = (N + kGemmBN - 1) / kGemmBN;
    if (rope && rope_heads > 0 && rope->rot_dim > 0) {
        P.rope = *rope;
        P.pos = pos;
        P.rope_heads = rope_heads;
    }
    const long long total = static_cast<long long>(P.m_tiles) * (P.n_tiles + (N2 > 0 ? 1 : 0));
    const int grid = static_cast<int>(total < gemm_sm_count() ? total : gemm_sm_count());
    cudaError_t err = cudaFuncSetAttribute(gemm_bf16_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kGemmSmemBytes);
    if (err == cudaSuccess)
        err = launch_overlapped(gemm_bf16_kernel, dim3(grid), dim3(kGemmThreads), kGemmSmemBytes,
                                stream, tm_x, tm_w, tm_w2, P);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return SPARK_ERR_CUDA;
    }
    return SPARK_OK;
}

}  // namespace spark

extern "C" spark_status spark_attn_linear(const void *x, const void *w, void *y, int64_t M, int N,
                                          int K, uint32_t *device_status, void *stream) {
    using namespace spark;
    const spark_status st = check_linear(x, w, y, M, N, K, nullptr, nullptr, 0);
    if (st != SPARK_OK || M == 0) return st;
    if (!device_status) return SPARK_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(device_status) % 4 != 0) return SPARK_ERR_ALIGN;
    return launch_linear(x, w, y, M, N, K, nullptr, nullptr, 0,
                         reinterpret_cast<unsigned *>(device_status),
                         static_cast<cudaStream_t>(stream), nullptr, nullptr, 0);
}
