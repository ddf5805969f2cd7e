// tcg_internal.h -- definitions shared by the host runtime and the kernels of libtcg.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tcg {

// Tile shape of the persistent GEMM kernel (one CTA per SM).
constexpr int kBM = 128;               // rows of D per tile (MMA M, TMEM lanes)
constexpr int kBN = 256;               // columns of D per tile (MMA N, TMEM columns)
constexpr int kRowBytes = 128;         // one 128-byte swizzle row of K per stage
constexpr int kStages = 4;             // shared-memory ring depth
constexpr int kABytes = kBM * kRowBytes;           // 16 KiB per stage
constexpr int kBBytes = kBN * kRowBytes;           // 32 KiB per stage
constexpr int kStageBytes = kABytes + kBBytes;     // 48 KiB per stage
constexpr int kAccBufs = 2;            // TMEM accumulator double buffer
constexpr int kTmemCols = kAccBufs * kBN;          // 512 columns = all of TMEM
constexpr int kEpiWarps = 4;
constexpr int kThreads = 32 * (2 + kEpiWarps);     // producer, MMA, 4 epilogue warps
constexpr int kBarrierBytes = 256;
constexpr int kSmemBytes = kStages * kStageBytes + kBarrierBytes + 1024;  // + alignment slack

// Bits of the device error word (which bounded wait gave up).
constexpr uint32_t kErrProducer = 1u;    // producer waiting for a free stage
constexpr uint32_t kErrMmaFull = 2u;     // MMA waiting for operands
constexpr uint32_t kErrMmaAcc = 4u;      // MMA waiting for a free accumulator
constexpr uint32_t kErrEpilogue = 8u;    // epilogue waiting for a finished accumulator
constexpr uint32_t kErrDrain = 16u;      // end-of-kernel drain

enum OutKind { kOutF32 = 0, kOutF16 = 1, kOutBF16 = 2 };

struct GemmArgs {
    int m, n, k;
    int batch;
    int num_m_tiles, num_n_tiles, num_k_blocks;
    int total_tiles;
    int group_m;               // tile rasterisation: group of m-tiles walked together
    int a_kmajor, b_kmajor;    // operand majorness in global memory
    int a_bcast, b_bcast;      // batch stride 0: always batch coordinate 0
    int is_tf32;               // kind::tf32 (else kind::f16)
    int k_per_block;           // K elements per stage: 64 (16-bit) or 32 (TF32)
    int mn_box;                // M/N elements per 128-byte run: 64 or 32
    uint32_t idesc;            // tcgen05 instruction descriptor
    float alpha, beta;
    const void *C;
    void *D;
    int64_t ldc, strideC;
    uint32_t *err;
    unsigned long long wait_limit_ns;
    int fault_inject;
};

// Launchers (tcg_kernels.cu).  Return the launch's cudaError_t.
cudaError_t launch_gemm(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmArgs &a,
                        int out_kind, int grid, cudaStream_t s);
cudaError_t launch_scale(void *D, const void *C, int m, int n, int64_t ldc, int64_t strideC,
                         int batch, float beta, int out_kind, int grid, cudaStream_t s);
cudaError_t launch_tf32_pack(const void *in, int64_t ld, int64_t stride_in, int in_kmajor,
                             int rows, int k, int batch, void *out, int64_t ld_out,
                             int64_t stride_out, int grid, cudaStream_t s);

}  // namespace tcg
