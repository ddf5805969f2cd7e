// tcg_internal.h -- definitions shared by the host runtime and the kernels of libtcg.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tcg {

// Tile shape of the persistent GEMM kernel (one CTA per SM).  With a CTA pair
// (cta_group::2) a tile is 256 x BN: each CTA of the pair holds 128 rows of A and BN / 2
// rows of B per stage and 128 rows of the accumulator; with a single CTA a tile is
// 128 x BN and the CTA holds all BN rows of B.  BN is 256, or 128 for problems too small
// to fill the GPU (twice the tiles: the epilogue of a lone tile is spread over twice the
// SMs; SM-pair kernel with FP16/BF16 inputs only).
constexpr int kBM = 128;               // rows of D per CTA (MMA M per CTA, TMEM lanes)
constexpr int kBN = 256;               // columns of D per tile (MMA N, TMEM columns)
constexpr int kBNNarrow = 128;         // the narrow tile width
constexpr int kRowBytes = 128;         // one 128-byte swizzle row of K
constexpr int kDepth = 1;              // 128-byte K rows per operand row and stage
constexpr int kABytes = kBM * kRowBytes;           // 16 KiB: A for one K row
constexpr int kTmemCols = 512;         // all of TMEM: 512 / BN accumulators (2 or 4)
constexpr int kMaxAccBufs = kTmemCols / kBNNarrow;
constexpr int kEpiWarps = 8;           // two warps per TMEM lane quarter
constexpr int kThreads = 32 * (2 + kEpiWarps);     // producer, MMA, 8 epilogue warps
// Shared memory: operand ring + epilogue staging = kDataBytes.  Epilogue staging: each
// half of the epilogue (4 warps, 128 rows) owns CBUF buffers (2 when C is not read) of
// one 128-row chunk of D (16 FP32 or 32 16-bit columns: 8 KiB; in the CBUF = 4 variant
// three buffers of 32 FP32 or 64 16-bit columns, 16 KiB -- see epi_chunk_bytes),
// loaded with C by TMA (buffers - 1) chunks ahead when beta != 0 and written back by TMA.
// Four buffers (and a shorter ring) pay off when
// the epilogue's C/D traffic outweighs the main loop: K bytes per operand row <= 1024 x
// D's element size (measured on 16384 x 4096 and batched 256 x 256 problems).
constexpr int kDataBytes = 224 * 1024;
constexpr int kEpiChunkBytes = 8 * 1024;
constexpr int kBarrierBytes = 512;
constexpr int kSmemBytes = kDataBytes + kBarrierBytes + 1024;  // + alignment slack
// Bytes and columns of one epilogue chunk.  The CBUF = 4 variant (short K: the epilogue's
// C/D traffic outweighs the main loop) stages 16 KiB chunks, 64 16-bit or 32 FP32 columns
// -- half the chunks per tile, so half the per-chunk barriers, proxy fences and TMA
// operations (measured on GB300: 512 batched 256^3 FP16 products, beta = 0.5, back to
// back, 51.8 -> 49.0 us with four such buffers; the 256^3 FP16 -> FP32 product, beta = 1,
// 14.3 -> 13.6-13.9 us; 16 KiB chunks in every variant slowed a 4096^3 FP16 -> FP16
// product, beta = 1, from 94 to 99 us through its shorter ring).  Every tensor map of D
// (or of the tail partial sums) that such a kernel stores through has a box this wide.
__host__ __device__ constexpr int epi_chunk_bytes(int out_bytes, int c_bufs)
{
    (void)out_bytes;
    return c_bufs == 4 ? 2 * kEpiChunkBytes : kEpiChunkBytes;
}
__host__ __device__ constexpr int epi_cols(int out_bytes, int c_bufs)
{
    return epi_chunk_bytes(out_bytes, c_bufs) / (kBM * out_bytes);
}

// One ring stage holds kDepth 128-byte rows of K for every operand row: K = 64 FP16/BF16,
// 32 TF32 or 128 FP8 elements (32 KiB a stage for a CTA of a pair, six stages).  What
// the tensor core sees depends on how many bytes are on their way when a stage is
// freed: with S stages of b bytes, (S - 2) * b of margin cover the load latency, so six
// stages of 32 KiB beat three of 64 KiB (measured per SM cycle, 8192^3 FP16: 96% of the
// MMA issue rate against 91-94%).  M/N-major tiles must still arrive in 16 KiB boxes:
// one box per 64-row chunk (8 KiB) starved the tensor core (82-90%), so whole-chunk
// operands use a 4-D view that brings a tile's chunks in one box (OperandMode kMN4).
template <int CG, int CBUF, int BN = kBN, int CHUNK = kEpiChunkBytes>
struct TileCfg {
    // CBUF 4 with its 16 KiB chunks keeps three of them, so that the ring
    // holds a whole K = 256 tile (four stages): batched 256^3 FP16, back to back 49.0 ->
    // 47-48 us, L2 flushed 59.4 -> 57.3 us.
    static constexpr int kEpiBufs = CBUF ? ((CBUF == 4 && CHUNK > kEpiChunkBytes) ? 3 : CBUF) : 2;
    static constexpr int kEpiBytes = 2 * kEpiBufs * CHUNK;   // 32, 64 or 96 KiB
    static constexpr int kRingBytes = kDataBytes - kEpiBytes;         // 192, 160 or 128 KiB
    static constexpr int kBRows = BN / CG;                   // B rows loaded per CTA
    static constexpr int kAStage = kABytes * kDepth;         // 16 KiB
    static constexpr int kBStage = kBRows * kRowBytes * kDepth;   // 16 KiB (pair), 32 KiB
    static constexpr int kStageBytes = kAStage + kBStage;    // 32 KiB (pair), 48 KiB (1 CTA)
    static constexpr int kStages = kRingBytes / kStageBytes; // pair: 6, 5 or 4; 1 CTA: 4 or 3
    static constexpr int kTileM = kBM * CG;                  // rows of D per tile
    static constexpr int kAccBufs = kTmemCols / BN;          // TMEM accumulators (2 or 4)
};

// Bits of the device error word (which bounded wait gave up).
constexpr uint32_t kErrProducer = 1u;    // producer waiting for a free stage
constexpr uint32_t kErrMmaFull = 2u;     // MMA waiting for operands
constexpr uint32_t kErrMmaAcc = 4u;      // MMA waiting for a free accumulator
constexpr uint32_t kErrEpilogue = 8u;    // epilogue waiting for a finished accumulator
constexpr uint32_t kErrDrain = 16u;      // end-of-kernel drain
constexpr uint32_t kErrConvert = 32u;    // producer waiting for in-kernel TF32 rounding

enum OutKind { kOutF32 = 0, kOutF16 = 1, kOutBF16 = 2 };

// MMA kind (operand formats): kind::f16 (FP16/BF16, K = 16 per instruction),
// kind::tf32 (K = 8), kind::f8f6f4 with E4M3/E5M2 (K = 32).  Every kind reads 32 bytes
// of K per instruction.  kKindTF32x3 is kind::tf32 on two words per operand (x = hi +
// lo): four operand tiles per stage and three products per K slice into one accumulator.
// kKindTF32R / kKindTF32x3R are kKindTF32 / kKindTF32x3 with the TF32 rounding (the
// two-word split) done inside the GEMM kernel (see the cv_* arguments) instead of by the
// separate pre-pass kernels.
enum MmaKind {
    kKindF16 = 0, kKindTF32 = 1, kKindF8 = 2, kKindTF32x3 = 3, kKindTF32R = 4, kKindTF32x3R = 5
};

// How an operand tile sits in global and shared memory (128-byte swizzle throughout).
//   kK:   K contiguous.  3-D map {K, rows, batch}, box {one 128-byte row of K, rows};
//         a stage holds kDepth such boxes one after the other (rows x 128 B each);
//         inside a box, 8-row groups are 1 KiB apart.
//   kMN:  M/N contiguous, rows not a multiple of c = 128 bytes / element size (64 for
//         16-bit operands, 128 for FP8; TF32 operands are always made K-major).  3-D map
//         {rows, K, batch}, box {c, kDepth 128-byte rows of K}; a stage holds one box per
//         c-element chunk of rows, chunk after chunk, each covering the stage's K range.
//   kMN4: M/N contiguous, rows a multiple of c.  4-D map {c, K, rows / c, batch}, box
//         {c, kDepth 128-byte rows of K, chunks of the tile}: the same shared-memory
//         layout as kMN from one box.
enum OperandMode { kK = 0, kMN = 1, kMN4 = 2 };

struct GemmArgs {
    int m, n, k;
    int batch;
    int num_m_tiles, num_n_tiles, num_k_blocks;   // K blocks of kDepth * k_row elements
    int total_tiles;           // work units: tiles x k_splits
    int k_splits;              // K ranges per tile (1: no split)
    int kb_per_split;          // K blocks per range (the last one may be shorter)
    int full_units;            // units [0, full_units) as above; then the split tail tiles
    int tail_splits;           // K ranges of each tail tile (1: no tail tiles)
    int tail_kb_per_split;     // K blocks per tail range
    int group_m;               // tile rasterisation: group of m-tiles walked together
    int a_mode, b_mode;        // OperandMode of A and B
    int a_bcast, b_bcast;      // batch stride 0: always batch coordinate 0
    int a_once, b_once;        // every element read by one tile only: L2 evict_first loads
    int kind;                  // MmaKind
    int k_row;                 // K elements per 128-byte row: 64, 32 (TF32), 128 (FP8)
    uint32_t idesc;            // tcgen05 instruction descriptor
    float alpha, beta;
    const void *C;
    void *D;
    int64_t ldc, strideC;
    uint32_t *err;
    unsigned long long wait_limit_ns;
    int fault_inject;
    int c_bufs;                // 0 (beta == 0), 2 or 4: epilogue variant (see TileCfg)
    // Clock probe (nullptr: off): every CTA adds the SM cycles (clock64) and nanoseconds
    // (globaltimer) it ran for to clk[0] and clk[1], so clk[0] / clk[1] is the SM clock
    // the kernel actually ran at.
    unsigned long long *clk;
    // TF32 rounding inside the GEMM kernel (kKindTF32R).  Index 0 is op(A), 1 is op(B).
    // The kernel writes the same rounded K-major copies the pre-pass would (element (r, q)
    // of batch entry b at cv_dst[x] + b * cv_dstride[x] + r * cv_kp + q), from the raw
    // FP32 operand (element (r, q) at cv_src[x] + b * cv_stride[x] + (cv_kmajor[x] ?
    // q + r * cv_ld[x] : r + q * cv_ld[x])).  The copies are cut into items: (operand,
    // batch entry, panel of cv_panel_rows[x] rows -- the tile rows of that operand --, chunk
    // of cv_kc K elements), item index cv_base[x] + (b * cv_panels[x] + panel) * cv_chunks
    // + chunk; and each item into cv_subs[x] sub-units of kCvRows rows x kCvK elements of
    // K.  cv_cnt holds three arrays of counters, zeroed before the launch: sub-units
    // claimed per item [cv_items], sub-units done per item [cv_items], and sub-units done
    // per panel [cv_panels_total] (panel index cv_pbase[x] + b * cv_panels[x] + panel).
    const void *cv_src[2];
    void *cv_dst[2];
    void *cv_dst_lo[2];        // two-word split: the low words, in the same layout
    int64_t cv_ld[2], cv_stride[2], cv_dstride[2];
    int64_t cv_kp;
    int cv_kmajor[2];
    int cv_rows[2];
    int cv_panel_rows[2];
    int cv_panels[2];
    int cv_subs[2];
    int cv_base[2], cv_pbase[2];
    int cv_kc, cv_chunks, cv_kb_per_chunk;
    int cv_items;
    uint32_t *cv_cnt;
};

// Sub-unit of the in-kernel TF32 rounding: 64 rows x 128 K elements (32 KiB of FP32).
constexpr int kCvRows = 64;
constexpr int kCvK = 128;

// Tile t -> (batch b, m-tile mt, n-tile nt) with grouped rasterisation.
__host__ __device__ inline void raster(const GemmArgs &p, int t, int &b, int &mt, int &nt)
{
    const int per_batch = p.num_m_tiles * p.num_n_tiles;
    b = t / per_batch;
    const int r = t - b * per_batch;
    const int span = p.group_m * p.num_n_tiles;
    const int g = r / span;
    const int first_m = g * p.group_m;
    const int gsize = p.num_m_tiles - first_m < p.group_m ? p.num_m_tiles - first_m : p.group_m;
    const int in_g = r - g * span;
    mt = first_m + in_g % gsize;
    nt = in_g / gsize;
}


// Tail split (FP32 output only): when the tiles fill whole waves of the SM pairs plus a
// partial last wave, the tiles of that partial wave (or of it and the wave before) are
// cut into `splits` K ranges whose partial sums go to tile-sized FP32 slices, and
// launch_tail_reduce adds them in range order and applies alpha and beta.  Each
// candidate (rest = tiles % clusters or that plus one wave; 2, 3 or 4 ranges) predicts
// full / clusters + ceil(rest * splits / clusters) / splits tile times against the
// unsplit ceil(tiles / clusters); only half of the predicted saving is counted (a partial
// wave runs on fewer SMs, which clock higher under the power cap: measured on 8192^3
// and TF32 4096 x 4096 x 16384 GEMMs).  The cost is a reduction launch (3 us) reading
// the partial sums and C and writing D (rest * (splits + 2) tiles of bytes at ~4 TB/s).
// The plan with the largest net saving is taken if it is positive; tile_us is the time
// of one whole tile.
struct TailPlan {
    int64_t full_tiles;        // tiles [0, full_tiles) whole
    int splits;                // 1: no tail split
    int kb_per_split;
};
inline TailPlan tail_plan(int64_t tiles, int num_k_blocks, int clusters, double tile_us,
                          double tile_bytes)
{
    TailPlan pl{tiles, 1, num_k_blocks};
    if (clusters <= 0 || tiles <= clusters || tiles % clusters == 0)
        return pl;
    const int64_t waves = (tiles + clusters - 1) / clusters;
    double best = 0.0;
    for (int c = 0; c < 2; ++c) {
        const int64_t rest = tiles % clusters + c * static_cast<int64_t>(clusters);
        if (rest >= tiles)
            break;
        const int64_t full = tiles - rest;
        for (int s = 2; s <= 4; ++s) {
            if (num_k_blocks < 2 * s)
                break;
            const int64_t tail_waves = (rest * s + clusters - 1) / clusters;
            const double t = static_cast<double>(full / clusters) +
                             static_cast<double>(tail_waves) / s;
            const double saved_us = 0.5 * (static_cast<double>(waves) - t) * tile_us;
            const double cost_us = 3.0 + static_cast<double>(rest * (s + 2)) * tile_bytes / 4.0e6;
            if (saved_us - cost_us > best) {
                best = saved_us - cost_us;
                pl.full_tiles = full;
                pl.splits = s;
            }
        }
    }
    if (pl.splits > 1) {
        pl.kb_per_split = (num_k_blocks + pl.splits - 1) / pl.splits;
        pl.splits = (num_k_blocks + pl.kb_per_split - 1) / pl.kb_per_split;
    }
    return pl;
}

// K splitting for problems with few tiles ("split-K"): each tile's K blocks are cut into
// k_splits ranges of kb_per_split blocks, every (tile, range) is a work unit whose FP32
// accumulator goes to a partial-sum workspace (slice b * k_splits + s), and
// launch_splitk_reduce adds the slices in range order and applies alpha, beta and the
// output rounding.  Split only when the tiles fill less than half of the clusters, with
// at least kMinSplitBlocks K blocks per range and at most kMaxSplits ranges; none of the
// ranges is empty.
constexpr int kMinSplitBlocks = 8;
constexpr int kMaxSplits = 64;
struct SplitPlan {
    int splits;
    int kb_per_split;
};
inline SplitPlan split_plan(int64_t tiles, int num_k_blocks, int clusters, int forced)
{
    SplitPlan pl{1, num_k_blocks};
    int s;
    if (forced >= 1) {
        s = forced;
    } else {
        if (tiles <= 0 || tiles * 2 > clusters)
            return pl;
        s = static_cast<int>(clusters / tiles);
        if (s > num_k_blocks / kMinSplitBlocks)
            s = num_k_blocks / kMinSplitBlocks;
    }
    if (s > kMaxSplits)
        s = kMaxSplits;
    if (s > num_k_blocks)
        s = num_k_blocks;
    if (s < 2)
        return pl;
    pl.kb_per_split = (num_k_blocks + s - 1) / s;
    pl.splits = (num_k_blocks + pl.kb_per_split - 1) / pl.kb_per_split;
    return pl;
}

// Launchers (tcg_kernels.cu).  Return the launch's cudaError_t.
// cta_group: 1 (128x256 tiles, one CTA) or 2 (256x256 tiles, CTA pairs; grid even).
// tmD maps D (= C) as {m, n, batch} with box {128, epi_cols(out bytes), 1}, no swizzle.
// tmW maps the tail partial sums (tile_m x 256 x slices FP32), used only when
// a.tail_splits > 1 (any valid map otherwise).
// bn: the tile width (kBN, or kBNNarrow where gemm_has_narrow says a variant exists).
// tmA2 / tmB2: the low words of A and B for kKindTF32x3 (tmA / tmB for the high words);
// nullptr for the other kinds.
cudaError_t launch_gemm(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmD,
                        const CUtensorMap &tmW, const GemmArgs &a, int out_kind, int cta_group,
                        int bn, int grid, cudaStream_t s, const CUtensorMap *tmA2 = nullptr,
                        const CUtensorMap *tmB2 = nullptr);
// Whether a narrow-tile (kBNNarrow) variant of the GEMM kernel exists for this launch.
bool gemm_has_narrow(int cta_group, int kind);
// D (FP32) of the split tail tiles from their partial sums W (see tcg_tail_reduce_kernel).
cudaError_t launch_tail_reduce(const float *W, int tail_tiles, int tile_m, const GemmArgs &a,
                               int grid, cudaStream_t s);
// Largest number of CTAs of the GEMM kernel that can be resident at once.
int gemm_max_resident_ctas(int cta_group, int num_sms);
cudaError_t launch_scale(void *D, const void *C, int m, int n, int64_t ldc, int64_t strideC,
                         int batch, float beta, int out_kind, int grid, cudaStream_t s);
// D[b] = alpha * (W[b*splits] + W[b*splits + 1] + ... in that order, FP32) + beta * C[b]
// (fma in FP32 when beta != 0), rounded to the output type; W slices are m x n FP32,
// column-major with leading dimension ldw and slice stride ldw * n.  C is D (in place).
cudaError_t launch_splitk_reduce(const float *W, int64_t ldw, int splits, int m, int n, int batch,
                                 float alpha, float beta, void *D, int64_t ldc, int64_t strideC,
                                 int out_kind, int grid, cudaStream_t s);
// Round FP32 -> TF32 (nearest even).  The tensor core takes TF32 operands K-major only
// and truncates the low 13 bits of FP32 input, so every TF32 operand gets a rounded,
// K-major copy: launch_tf32_round keeps an operand that is already K-major (rows = K,
// cols = M or N; ld, ld_out and strides multiples of 4 elements, 16-byte aligned
// pointers); launch_tf32_transpose_round turns an M/N-major one (rows = M or N along
// the contiguous dimension) into a K-major copy with leading dimension ld_out.
// out_lo (nullable): also write the low word of the two-word TF32 split (out = high
// word) in the same layout as out.
cudaError_t launch_tf32_round(const void *in, int64_t ld, int64_t stride_in, int64_t rows,
                              int64_t cols, int64_t batch, void *out, int64_t ld_out,
                              int64_t stride_out, void *out_lo, cudaStream_t s);
cudaError_t launch_tf32_transpose_round(const void *in, int64_t ld, int64_t stride_in,
                                        int64_t rows, int64_t k, int64_t batch, void *out,
                                        int64_t ld_out, int64_t stride_out, void *out_lo,
                                        cudaStream_t s);
// Round FP32 -> TF32 into a K-major packed copy (used by tcg_gemm_tf32_noalloc).
cudaError_t launch_tf32_pack(const void *in, int64_t ld, int64_t stride_in, int in_kmajor,
                             int rows, int k, int batch, void *out, int64_t ld_out,
                             int64_t stride_out, int grid, cudaStream_t s);

}  // namespace tcg
