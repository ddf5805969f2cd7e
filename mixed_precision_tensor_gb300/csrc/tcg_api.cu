// tcg_api.cu -- host runtime and C ABI of libtcg (declared in include/tcg.h).
//
// Order of work in a GEMM call:
//   1. argument checks (pure host code, no CUDA call): the GemmEx argument rules of
//      "Programming Tensor Cores in CUDA 9", section "如何在 cuBLAS 中使用张量核",
//      restated for TMA (16-byte aligned pointers and leading dimensions);
//   2. device binding on first use (compute capability 10.3, SM count, error word);
//   3. dispatch: k == 0 or alpha == 0 -> D = beta*C kernel; TF32 -> round-and-pack
//      kernels into the workspace, then the GEMM kernel on the packed copies;
//      FP16/BF16 -> the GEMM kernel straight on the caller's operands;
//   4. tensor maps (cached per pointer/shape/stride/type) and a persistent grid of
//      min(tiles, SMs) CTAs on the handle's stream.

#include <cstdlib>
#include <mutex>
#include <cstring>
#include <new>

#include "tcg.h"
#include "tcg_internal.h"

using namespace tcg;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
constexpr int kMapCacheSize = 32;
constexpr int kPtrCacheSize = 16;

struct MapKey {
    const void *ptr;
    int dtype;
    int rank;
    int swizzle;
    uint64_t dims[5];
    uint64_t strides[4];
    uint32_t box[5];
    bool operator==(const MapKey &o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};

constexpr int kHostChunks = 16;     // chunks of a host-buffer call (events per handle)
constexpr int kHostPanels = 4;      // chunks of the panel / batch-group split

struct MapEntry {
    MapKey key;
    CUtensorMap map;
    bool valid;
};

}  // namespace

struct tcgContext {
    int device = -1;
    int num_sms = 0;
    cudaStream_t stream = nullptr;
    uint32_t *d_err = nullptr;
    unsigned long long *d_clk = nullptr;   // clock probe counters (tcg_set_clock_probe)
    bool clk_on = false;
    void *ws_user = nullptr;
    size_t ws_user_bytes = 0;
    void *ws_own = nullptr;
    size_t ws_own_bytes = 0;
    unsigned long long wait_limit_ns = kDefaultWaitNs;
    int fault_inject = 0;
    uint64_t launches = 0;
    uint32_t last_err_bits = 0;
    int cta_group = 2;
    int group_m = 0;           // 0: choose per problem
    int split_k = 0;           // 0: choose per problem, 1: never split, >= 2: that many ranges
    int tile_n = 0;            // 0: choose per problem, or kBN / kBNNarrow
    int tf32_round = 0;        // TF32 rounding: 0 choose, 1 pre-pass kernels, 2 in the GEMM
    // Host-buffer calls: device copies of A, B, C (grown on demand) and two copy streams.
    void *stage_buf[3] = {nullptr, nullptr, nullptr};
    size_t stage_bytes[3] = {0, 0, 0};
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t ev_in[kHostChunks] = {}, ev_out[kHostChunks] = {};
    int max_ctas[3] = {0, 0, 0};
    bool used = false;
    EncodeTiledFn encode = nullptr;
    MapEntry cache[kMapCacheSize];
    int cache_next = 0;
    const void *ptr_ok[kPtrCacheSize] = {};   // pointers already found to be device memory
    int ptr_next = 0;
};

namespace {

int elem_size(tcgDataType_t t)
{
    return t == TCG_R_32F ? 4 : ((t == TCG_R_8F_E4M3 || t == TCG_R_8F_E5M2) ? 1 : 2);
}

bool is_fp8(int t) { return t == TCG_R_8F_E4M3 || t == TCG_R_8F_E5M2; }

bool valid_type(int t)
{
    return t == TCG_R_16F || t == TCG_R_16BF || t == TCG_R_32F || is_fp8(t);
}

int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Problem {
    tcgOp_t transa, transb;
    int64_t m, n, k;
    float alpha, beta;
    const void *A; tcgDataType_t Atype; int64_t lda; int64_t strideA;
    const void *B; tcgDataType_t Btype; int64_t ldb; int64_t strideB;
    void *C; tcgDataType_t Ctype; int64_t ldc; int64_t strideC;
    int64_t batch;
    tcgComputeType_t compute;
    bool batched;
    bool staged = false;       // A, B, C are the handle's own staging buffers (host-buffer calls)
};

// Pure host argument checks: no CUDA call is made before they pass.
tcgStatus_t check_args(const Problem &p)
{
    if ((p.transa != TCG_OP_N && p.transa != TCG_OP_T) ||
        (p.transb != TCG_OP_N && p.transb != TCG_OP_T))
        return TCG_STATUS_INVALID_VALUE;
    if (!valid_type(p.Atype) || !valid_type(p.Btype) || !valid_type(p.Ctype))
        return TCG_STATUS_INVALID_VALUE;
    if (p.compute != TCG_COMPUTE_32F && p.compute != TCG_COMPUTE_32F_FAST_TF32 &&
        p.compute != TCG_COMPUTE_32F_3XTF32)
        return TCG_STATUS_INVALID_VALUE;
    if (p.m < 0 || p.n < 0 || p.k < 0 || p.batch < 0)
        return TCG_STATUS_INVALID_VALUE;
    // Supported (A/B, compute, C) combinations.
    if (p.Atype != p.Btype || is_fp8(p.Ctype))
        return TCG_STATUS_NOT_SUPPORTED;
    if (p.Atype == TCG_R_32F) {
        if (p.compute == TCG_COMPUTE_32F || p.Ctype != TCG_R_32F)
            return TCG_STATUS_NOT_SUPPORTED;
    } else if (is_fp8(p.Atype)) {
        if (p.compute != TCG_COMPUTE_32F)       // FP32, FP16 or BF16 output
            return TCG_STATUS_NOT_SUPPORTED;
    } else {
        if (p.compute != TCG_COMPUTE_32F)
            return TCG_STATUS_NOT_SUPPORTED;
        if (p.Ctype != TCG_R_32F && p.Ctype != p.Atype)
            return TCG_STATUS_NOT_SUPPORTED;
    }
    // Leading dimensions (BLAS rules), then the 16-byte TMA rule.
    const int64_t a_rows = p.transa == TCG_OP_N ? p.m : p.k;
    const int64_t b_rows = p.transb == TCG_OP_N ? p.k : p.n;
    if (p.lda < max64(1, a_rows) || p.ldb < max64(1, b_rows) || p.ldc < max64(1, p.m))
        return TCG_STATUS_INVALID_VALUE;
    const int ea = elem_size(p.Atype), ec = elem_size(p.Ctype);
    if ((p.lda * ea) % 16 || (p.ldb * ea) % 16 || (p.ldc * ec) % 16)
        return TCG_STATUS_INVALID_VALUE;
    if (p.batched) {
        if (p.strideA < 0 || p.strideB < 0 || p.strideC < 0)
            return TCG_STATUS_INVALID_VALUE;
        if ((p.strideA * ea) % 16 || (p.strideB * ea) % 16 || (p.strideC * ec) % 16)
            return TCG_STATUS_INVALID_VALUE;
        if (p.strideC == 0 && p.batch > 1)
            return TCG_STATUS_INVALID_VALUE;
    }
    // Limits of the kernels' 32-bit tile and TMA coordinates.
    const int64_t lim = (int64_t(1) << 31) - 1;
    if (p.m > lim || p.n > lim || p.k > lim || p.batch > lim)
        return TCG_STATUS_NOT_SUPPORTED;
    if (p.m == 0 || p.n == 0 || p.batch == 0)
        return TCG_STATUS_SUCCESS;
    const bool reads_ab = p.k > 0 && p.alpha != 0.0f;
    if (!p.C || !aligned16(p.C))
        return TCG_STATUS_INVALID_VALUE;
    if (reads_ab && (!p.A || !p.B || !aligned16(p.A) || !aligned16(p.B)))
        return TCG_STATUS_INVALID_VALUE;
    const int64_t tiles_m = (p.m + kBM - 1) / kBM, tiles_n = (p.n + kBN - 1) / kBN;
    if (tiles_m * tiles_n * p.batch > lim)
        return TCG_STATUS_NOT_SUPPORTED;
    return TCG_STATUS_SUCCESS;
}

tcgStatus_t bind_device(tcgContext *h)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return TCG_STATUS_NOT_INITIALIZED;
    }
    if (h->device >= 0) {
        return dev == h->device ? TCG_STATUS_SUCCESS : TCG_STATUS_INVALID_VALUE;
    }
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return TCG_STATUS_NOT_INITIALIZED;
    }
    if (major != 10 || minor != 3)
        return TCG_STATUS_ARCH_MISMATCH;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        cudaGetLastError();
        return TCG_STATUS_NOT_INITIALIZED;
    }
    uint32_t *err = nullptr;
    if (cudaMalloc(&err, sizeof(uint32_t)) != cudaSuccess) {
        cudaGetLastError();
        return TCG_STATUS_ALLOC_FAILED;
    }
    if (cudaMemset(err, 0, sizeof(uint32_t)) != cudaSuccess) {
        cudaFree(err);
        cudaGetLastError();
        return TCG_STATUS_EXECUTION_FAILED;
    }
    h->encode = reinterpret_cast<EncodeTiledFn>(fn);
    h->d_err = err;
    h->num_sms = sms;
    h->device = dev;
    return TCG_STATUS_SUCCESS;
}

// The device-buffer calls hand their pointers to TMA and to plain kernel loads and
// stores, where a host address would fault the GPU rather than fail the call.  So each
// pointer must be device memory of the bound device (cudaMalloc, stream-ordered pool or
// VMM allocation); pageable, pinned (cudaHostAlloc) and managed memory are rejected.
// The query is a pure lookup, made in relaxed capture mode so that a call being
// captured into a CUDA graph cannot have it counted as an unsafe call.
tcgStatus_t device_ptr_ok(int dev, const void *p)
{
    cudaPointerAttributes at;
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    const bool swapped = cudaThreadExchangeStreamCaptureMode(&mode) == cudaSuccess;
    const cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (swapped)
        cudaThreadExchangeStreamCaptureMode(&mode);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return TCG_STATUS_INVALID_VALUE;
    }
    return at.type == cudaMemoryTypeDevice && at.device == dev ? TCG_STATUS_SUCCESS
                                                                : TCG_STATUS_INVALID_VALUE;
}

// device_ptr_ok with a small per-handle cache of the pointer values that passed, so a
// repeated call costs no driver query.
tcgStatus_t device_ptr_cached(tcgContext *h, const void *p)
{
    for (int i = 0; i < kPtrCacheSize; ++i)
        if (h->ptr_ok[i] == p)
            return TCG_STATUS_SUCCESS;
    const tcgStatus_t st = device_ptr_ok(h->device, p);
    if (st == TCG_STATUS_SUCCESS) {
        h->ptr_ok[h->ptr_next] = p;
        h->ptr_next = (h->ptr_next + 1) % kPtrCacheSize;
    }
    return st;
}

// The operands a device-buffer call touches: C always, A and B when the product is formed.
tcgStatus_t check_ptrs(tcgContext *h, const Problem &p)
{
    tcgStatus_t st = device_ptr_cached(h, p.C);
    if (st == TCG_STATUS_SUCCESS && p.k > 0 && p.alpha != 0.0f) {
        st = device_ptr_cached(h, p.A);
        if (st == TCG_STATUS_SUCCESS)
            st = device_ptr_cached(h, p.B);
    }
    return st;
}

CUtensorMapDataType map_type(tcgDataType_t t)
{
    switch (t) {
    case TCG_R_16F: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    case TCG_R_16BF: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    case TCG_R_8F_E4M3:
    case TCG_R_8F_E5M2: return CU_TENSOR_MAP_DATA_TYPE_UINT8;   // raw bytes
    default: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    }
}

// Tiled map of rank 3 or 4 with 128-byte swizzle and zero fill out of range, cached
// per (pointer, type, dims, strides, box).
tcgStatus_t get_map(tcgContext *h, const void *ptr, tcgDataType_t t, int rank,
                    const uint64_t *dims, const uint64_t *strides, const uint32_t *box,
                    CUtensorMap *out, bool swizzle = true)
{
    MapKey key;
    std::memset(&key, 0, sizeof key);
    key.ptr = ptr;
    key.dtype = static_cast<int>(t);
    key.rank = rank;
    key.swizzle = swizzle ? 1 : 0;
    for (int i = 0; i < rank; ++i) {
        key.dims[i] = dims[i];
        key.box[i] = box[i];
        if (i < rank - 1)
            key.strides[i] = strides[i];
    }
    for (int i = 0; i < kMapCacheSize; ++i) {
        if (h->cache[i].valid && h->cache[i].key == key) {
            *out = h->cache[i].map;
            return TCG_STATUS_SUCCESS;
        }
    }
    alignas(64) CUtensorMap map;
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = h->encode(&map, map_type(t), static_cast<cuuint32_t>(rank),
                           const_cast<void *>(ptr), key.dims, key.strides, key.box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return TCG_STATUS_EXECUTION_FAILED;
    MapEntry &e = h->cache[h->cache_next];
    h->cache_next = (h->cache_next + 1) % kMapCacheSize;
    e.key = key;
    e.map = map;
    e.valid = true;
    *out = map;
    return TCG_STATUS_SUCCESS;
}

// Map for one operand as the kernel loads it (see OperandMode).  rows = M (for A) or
// N (for B); box_rows = the rows one CTA loads per stage (128 for A; 256 or 128 for B);
// k_row = K elements per 128-byte row.
tcgStatus_t operand_map(tcgContext *h, const void *ptr, tcgDataType_t t, bool kmajor,
                        int64_t rows, int64_t k, int64_t ld, int64_t stride, int64_t batch,
                        int box_rows, int k_row, bool *bcast, int *mode, CUtensorMap *out)
{
    const int es = elem_size(t);
    const bool bc = (batch > 1 && stride == 0);
    *bcast = bc;
    const uint64_t nb = bc ? 1 : static_cast<uint64_t>(batch);
    const uint64_t ldb = static_cast<uint64_t>(ld) * es;
    const uint64_t outer = kmajor ? rows : k;
    uint64_t bstride = static_cast<uint64_t>(stride) * es;
    if (nb == 1)
        bstride = ldb * outer;                  // unused; any legal value
    if (bstride == 0)
        bstride = 16;
    if (kmajor) {
        *mode = kK;
        const uint64_t dims[3] = {static_cast<uint64_t>(k), static_cast<uint64_t>(rows), nb};
        const uint64_t str[2] = {ldb, bstride};
        const uint32_t box[3] = {static_cast<uint32_t>(k_row), static_cast<uint32_t>(box_rows),
                                 1};
        return get_map(h, ptr, t, 3, dims, str, box, out);
    }
    // M/N-major with whole chunks: the 4-D view {c, K, rows / c, batch} brings all of a
    // tile's chunks in one box (chunk after chunk, each over the stage's K rows).
    const int c = 128 / es;
    if (rows % c == 0) {
        *mode = kMN4;
        const uint64_t dims[4] = {static_cast<uint64_t>(c), static_cast<uint64_t>(k),
                                  static_cast<uint64_t>(rows / c), nb};
        const uint64_t str[3] = {ldb, 128, bstride};
        const uint32_t box[4] = {static_cast<uint32_t>(c), static_cast<uint32_t>(kDepth * k_row),
                                 static_cast<uint32_t>(box_rows / c), 1};
        return get_map(h, ptr, t, 4, dims, str, box, out);
    }
    // M/N-major, ragged rows: one 3-D box per 128-byte chunk of rows (the 4-D view would
    // read the next column's elements into the last chunk instead of zeros).
    *mode = kMN;
    const uint64_t dims[3] = {static_cast<uint64_t>(rows), static_cast<uint64_t>(k), nb};
    const uint64_t str[2] = {ldb, bstride};
    const uint32_t box[3] = {static_cast<uint32_t>(128 / es), static_cast<uint32_t>(kDepth * k_row),
                             1};
    return get_map(h, ptr, t, 3, dims, str, box, out);
}

// Map of D (= C) for the epilogue: {m, n, batch}, box {128 rows, chunk columns, 1}, no
// swizzle; TMA loads of C zero-fill and TMA stores of D clip outside the matrix.
tcgStatus_t output_map(tcgContext *h, void *C, tcgDataType_t t, int64_t m, int64_t n,
                       int64_t ldc, int64_t strideC, int64_t batch, CUtensorMap *out,
                       int c_bufs = 0)
{
    const int es = elem_size(t);
    const uint64_t ldb = static_cast<uint64_t>(ldc) * es;
    uint64_t bstride = static_cast<uint64_t>(strideC) * es;
    if (batch <= 1 || bstride == 0)
        bstride = ldb * static_cast<uint64_t>(n);       // unused; any legal value
    const uint64_t dims[3] = {static_cast<uint64_t>(m), static_cast<uint64_t>(n),
                              static_cast<uint64_t>(batch < 1 ? 1 : batch)};
    const uint64_t str[2] = {ldb, bstride};
    const uint32_t box[3] = {static_cast<uint32_t>(kBM),
                             static_cast<uint32_t>(epi_cols(es, c_bufs)), 1};
    return get_map(h, C, t, 3, dims, str, box, out, false);
}

int out_kind(tcgDataType_t c)
{
    return c == TCG_R_32F ? kOutF32 : (c == TCG_R_16F ? kOutF16 : kOutBF16);
}

size_t tf32_ws_bytes(int64_t m, int64_t n, int64_t k, int64_t batch)
{
    const int64_t kp = (k + 3) / 4 * 4;
    const size_t a = ((size_t)(batch * m * kp) * 4 + 255) / 256 * 256;
    const size_t b = ((size_t)(batch * n * kp) * 4 + 255) / 256 * 256;
    return a + b;
}

// In-kernel TF32 rounding (kKindTF32R): the rounded copies are cut into items of
// kCvChunk K elements by one panel of tile rows (see GemmArgs::cv_*), with three
// counters per item and panel in the workspace after the copies.
constexpr int kCvChunk = 1024;
constexpr int64_t kMaxCvItems = int64_t(1) << 20;
struct CvPlan {
    int64_t items, panels;
    int panels_a, panels_b, chunks;
};
CvPlan cv_plan(int64_t m, int64_t n, int64_t k, int64_t nba, int64_t nbb, int rows_a, int rows_b)
{
    CvPlan c;
    const int64_t kp = (k + 3) / 4 * 4;
    c.chunks = static_cast<int>((kp + kCvChunk - 1) / kCvChunk);
    c.panels_a = static_cast<int>((m + rows_a - 1) / rows_a);
    c.panels_b = static_cast<int>((n + rows_b - 1) / rows_b);
    c.panels = nba * c.panels_a + nbb * c.panels_b;
    c.items = c.panels * c.chunks;
    return c;
}
size_t cv_ws_bytes(const CvPlan &c)
{
    return ((size_t)(2 * c.items + c.panels) * 4 + 255) / 256 * 256;
}

// Partial-sum workspace of a split-K call: batch * splits slices of round_up(m, 4) x n
// FP32 values.
size_t splitk_ws_bytes(int64_t m, int64_t n, int64_t batch, int splits)
{
    const int64_t ldw = (m + 3) / 4 * 4;
    return ((size_t)(batch * splits) * (size_t)(ldw * n) * 4 + 255) / 256 * 256;
}

// Output tiles of a problem with tiles of (128 cg) x bn.
int64_t tiles_of(int64_t m, int64_t n, int64_t batch, int cg, int bn)
{
    return ((m + kBM * cg - 1) / (kBM * cg)) * ((n + bn - 1) / bn) * batch;
}

// The K split the GEMM of this problem gets on handle h (see split_plan).
SplitPlan plan_for(tcgContext *h, int64_t m, int64_t n, int64_t k, int64_t batch, int es, int cg,
                   int bn = kBN)
{
    if (h->max_ctas[cg] == 0)
        h->max_ctas[cg] = gemm_max_resident_ctas(cg, h->num_sms);
    const int64_t k_block = static_cast<int64_t>(kDepth) * (128 / es);
    const int nkb = static_cast<int>((k + k_block - 1) / k_block);
    return split_plan(tiles_of(m, n, batch, cg, bn), nkb, h->max_ctas[cg] / cg, h->split_k);
}

// The tile width of a call (see kBNNarrow).  Automatic choice: the narrow tile when the
// 256-wide tiles would fill at most half of the SM pairs and K is split at neither width
// (a split already spreads such a problem over the GPU).
int tile_n_for(tcgContext *h, int64_t m, int64_t n, int64_t k, int64_t batch, int es, int cg,
               int kind)
{
    if (!gemm_has_narrow(cg, kind) || h->tile_n == kBN ||
        tiles_of(m, n, batch, cg, kBNNarrow) * kMaxSplits > INT32_MAX)
        return kBN;
    if (h->tile_n == kBNNarrow)
        return kBNNarrow;
    const SplitPlan wide = plan_for(h, m, n, k, batch, es, cg, kBN);
    const int64_t clusters = h->max_ctas[cg] / cg;
    if (wide.splits > 1 || clusters <= 0 || tiles_of(m, n, batch, cg, kBN) * 2 > clusters)
        return kBN;
    return plan_for(h, m, n, k, batch, es, cg, kBNNarrow).splits > 1 ? kBN : kBNNarrow;
}

// The tail split of an unsplit problem with FP32 output (see tail_plan); none otherwise.
// A K block (kDepth x 128 bytes of K for every row) keeps the tensor pipe 512 cycles per
// 128-byte row busy on either kernel variant; ~1.8 GHz is taken for the tile time.
TailPlan tail_for(tcgContext *h, int64_t m, int64_t n, int64_t k, int64_t batch, int es, int cg,
                  bool fp32_out, const SplitPlan &split, int bn = kBN, double mmas_per_slice = 1.0)
{
    const int64_t k_block = static_cast<int64_t>(kDepth) * (128 / es);
    const int nkb = static_cast<int>((k + k_block - 1) / k_block);
    const int64_t tiles = tiles_of(m, n, batch, cg, bn);
    if (!fp32_out || split.splits > 1 || h->split_k != 0 || bn != kBN)
        return TailPlan{tiles, 1, nkb};
    const double tile_us = nkb * 512.0 * kDepth * mmas_per_slice / 1.8e3;
    return tail_plan(tiles, nkb, h->max_ctas[cg] / cg, tile_us, 4.0 * kBM * cg * kBN);
}

// Device workspace of at least `need` bytes: the caller's (tcg_set_workspace) or one the
// handle grows with cudaMalloc.
tcgStatus_t acquire_ws(tcgContext *h, size_t need, void **ws)
{
    if (h->ws_user) {
        if (h->ws_user_bytes < need || device_ptr_cached(h, h->ws_user) != TCG_STATUS_SUCCESS)
            return TCG_STATUS_INVALID_VALUE;
        *ws = h->ws_user;
        return TCG_STATUS_SUCCESS;
    }
    if (h->ws_own_bytes < need) {
        if (h->ws_own) {
            cudaStreamSynchronize(h->stream);
            cudaFree(h->ws_own);
            h->ws_own = nullptr;
            h->ws_own_bytes = 0;
        }
        if (cudaMalloc(&h->ws_own, need) != cudaSuccess) {
            cudaGetLastError();
            h->ws_own = nullptr;
            return TCG_STATUS_ALLOC_FAILED;
        }
        h->ws_own_bytes = need;
    }
    *ws = h->ws_own;
    return TCG_STATUS_SUCCESS;
}

tcgStatus_t run(tcgContext *h, const Problem &p)
{
    tcgStatus_t st = check_args(p);
    if (st != TCG_STATUS_SUCCESS)
        return st;
    if (p.m == 0 || p.n == 0 || p.batch == 0)
        return TCG_STATUS_SUCCESS;
    st = bind_device(h);
    if (st != TCG_STATUS_SUCCESS)
        return st;
    if (!p.staged) {
        st = check_ptrs(h, p);
        if (st != TCG_STATUS_SUCCESS)
            return st;
    }
    h->used = true;
    const int ok = out_kind(p.Ctype);
    const int m = static_cast<int>(p.m), n = static_cast<int>(p.n), k = static_cast<int>(p.k);
    const int batch = static_cast<int>(p.batch);
    const int64_t strideC = p.batched ? p.strideC : 0;

    if (p.k == 0 || p.alpha == 0.0f) {
        const int64_t total = p.m * p.n * p.batch;
        int64_t blocks = (total + 255) / 256;
        const int64_t cap = static_cast<int64_t>(h->num_sms) * 8;
        if (blocks > cap) blocks = cap;
        cudaError_t e = launch_scale(p.C, p.C, m, n, p.ldc, strideC, batch, p.beta, ok,
                                     static_cast<int>(blocks), h->stream);
        h->launches += 1;
        return e == cudaSuccess ? TCG_STATUS_SUCCESS : TCG_STATUS_EXECUTION_FAILED;
    }

    // TF32 compute and the three-product split both run on rounded K-major copies.
    const bool split3 = p.compute == TCG_COMPUTE_32F_3XTF32;
    const bool tf32 = p.compute == TCG_COMPUTE_32F_FAST_TF32 || split3;
    const int cg = h->cta_group;
    const int es_k = tf32 ? 4 : elem_size(p.Atype);
    // The two-word split runs as one GEMM kernel with three products per K slice.
    const int kind = split3 ? kKindTF32x3
                            : (tf32 ? kKindTF32 : (is_fp8(p.Atype) ? kKindF8 : kKindF16));
    const int bn = tile_n_for(h, p.m, p.n, p.k, p.batch, es_k, cg, kind);
    const SplitPlan plan = plan_for(h, p.m, p.n, p.k, p.batch, es_k, cg, bn);
    const TailPlan tail = tail_for(h, p.m, p.n, p.k, p.batch, es_k, cg, p.Ctype == TCG_R_32F,
                                   plan, bn, split3 ? 3.0 : 1.0);
    const int64_t n_tiles_total = tiles_of(p.m, p.n, p.batch, cg, bn);
    const int64_t tail_tiles = tail.splits > 1 ? n_tiles_total - tail.full_tiles : 0;
    const size_t tf32_bytes = tf32 ? (split3 ? 2 : 1) * tf32_ws_bytes(p.m, p.n, p.k, p.batch) : 0;
    const size_t splitk_bytes = plan.splits > 1 ? splitk_ws_bytes(p.m, p.n, p.batch, plan.splits)
                                                : (tail_tiles ? (size_t)(tail_tiles * tail.splits) *
                                                                    (size_t)(kBM * cg * kBN) * 4
                                                              : 0);
    // TF32 rounding inside the GEMM kernel, or by the pre-pass kernels before it.
    const int64_t nba0 = (p.batched ? p.strideA : 0) == 0 ? 1 : p.batch;
    const int64_t nbb0 = (p.batched ? p.strideB : 0) == 0 ? 1 : p.batch;
    const CvPlan cvp = cv_plan(p.m, p.n, p.k, nba0, nbb0, kBM * cg, bn);
    // Rounding inside the GEMM kernel: always in mode 2, never in mode 1; by default only
    // for the two-word split with unsplit K of at least 6144.  Plain TF32 loses with it
    // (4096 x 4096 x 16384: 781 against 702 us per call): a tensor core fed at full rate
    // leaves the SM's shared-memory/L1 data path almost no room for the rounding's loads
    // and stores.  The split's three products per stage leave more, and it gains there
    // (GB300, same-box A/B with 1024-element items: 2048 x 2048 x 8192 +3.3%, 4096 x 4096
    // x 6144 +2.4%, 4096^3 and 8192 x 8192 x 4096 even, 4096 x 8192 x 2048 -0.9%; with
    // 512-element items 4096 x 4096 x 16384 +2.2% and 8192^3 +1.6%, then 2.1% and 0.7% more
    // with 1024; 1024 x 1024 x 16384, split K, -19%).
    const bool fuse_auto = split3 && plan.splits == 1 && p.k >= 6144;
    const bool fuse = tf32 && cvp.items <= kMaxCvItems &&
                      (h->tf32_round == 2 || (h->tf32_round == 0 && fuse_auto));
    const size_t cv_bytes = fuse ? cv_ws_bytes(cvp) : 0;
    void *ws = nullptr;
    if (tf32_bytes + splitk_bytes + cv_bytes > 0) {
        st = acquire_ws(h, tf32_bytes + splitk_bytes + cv_bytes, &ws);
        if (st != TCG_STATUS_SUCCESS)
            return st;
    }
    uint32_t *cv_cnt = fuse ? reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws) + tf32_bytes +
                                                           splitk_bytes)
                            : nullptr;
    float *W = splitk_bytes ? reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + tf32_bytes)
                            : nullptr;
    const int64_t ldw = (p.m + 3) / 4 * 4;
    const void *Aop = p.A, *Bop = p.B;
    const void *Alo = nullptr, *Blo = nullptr;
    bool a_kmajor = p.transa == TCG_OP_T;   // op(A) = A^T: K is A's contiguous dim
    bool b_kmajor = p.transb == TCG_OP_N;   // op(B) = B:   K is B's contiguous dim
    int64_t lda = p.lda, ldb = p.ldb;
    int64_t sA = p.batched ? p.strideA : 0, sB = p.batched ? p.strideB : 0;

    if (tf32) {
        // Round to TF32 (nearest even) into K-major copies of op(A) and op(B) in the
        // workspace (the tensor core takes TF32 operands K-major only and truncates the low
        // 13 bits of FP32 input): K-major operands are rounded in place order, M/N-major
        // ones transposed on the way.  The split also writes the low words (x - hi).
        const size_t one = tf32_ws_bytes(p.m, p.n, p.k, p.batch);
        const int64_t kp = (p.k + 3) / 4 * 4;
        uint8_t *Ak = static_cast<uint8_t *>(ws);
        uint8_t *Bk = Ak + ((size_t)(p.batch * p.m * kp) * 4 + 255) / 256 * 256;
        uint8_t *Akl = split3 ? Ak + one : nullptr;
        uint8_t *Bkl = split3 ? Bk + one : nullptr;
        // a batch stride of 0 (one operand shared by all batches) stays shared
        const int64_t nba = sA == 0 ? 1 : p.batch, nbb = sB == 0 ? 1 : p.batch;
        cudaError_t e;
        if (fuse) {
            // the GEMM kernel rounds the operands itself: only its counters start at zero
            e = cudaMemsetAsync(cv_cnt, 0, cv_bytes, h->stream);
        } else {
            e = a_kmajor
                ? launch_tf32_round(p.A, p.lda, sA, p.k, p.m, nba, Ak, kp, p.m * kp, Akl, h->stream)
                : launch_tf32_transpose_round(p.A, p.lda, sA, p.m, p.k, nba, Ak, kp, p.m * kp, Akl,
                                              h->stream);
            if (e == cudaSuccess)
                e = b_kmajor
                    ? launch_tf32_round(p.B, p.ldb, sB, p.k, p.n, nbb, Bk, kp, p.n * kp, Bkl,
                                        h->stream)
                    : launch_tf32_transpose_round(p.B, p.ldb, sB, p.n, p.k, nbb, Bk, kp, p.n * kp,
                                                  Bkl, h->stream);
            h->launches += 2;
        }
        if (e != cudaSuccess)
            return TCG_STATUS_EXECUTION_FAILED;
        Aop = Ak;
        Bop = Bk;
        Alo = Akl;
        Blo = Bkl;
        a_kmajor = b_kmajor = true;
        lda = ldb = kp;
        sA = sA == 0 ? 0 : p.m * kp;
        sB = sB == 0 ? 0 : p.n * kp;
    }

    const bool fp8 = is_fp8(p.Atype);
    const tcgDataType_t at = tf32 ? TCG_R_32F : p.Atype;
    const bool splitk = plan.splits > 1;
    // The GEMM kernel writes D -- or, split, the FP32 partial sums (slice b * splits + s).
    CUtensorMap tmD;
    // Four C buffers (one operand stage less; 16 KiB chunks for 16-bit outputs) when the
    // epilogue's C/D traffic outweighs the main loop: K bytes per row <= 1024 x D's element
    // size.  Split, the kernel writes raw partial sums (beta 0).
    const int c_bufs = (splitk || p.beta == 0.0f) ? 0
                     : (cg == 2 && k * es_k <= 1024 * elem_size(p.Ctype) ? 4 : 2);
    st = splitk ? output_map(h, W, TCG_R_32F, p.m, p.n, ldw, ldw * p.n, p.batch * plan.splits,
                             &tmD)
                : output_map(h, p.C, p.Ctype, p.m, p.n, p.ldc, strideC, p.batch, &tmD, c_bufs);
    if (st != TCG_STATUS_SUCCESS)
        return st;
    // Split tail tiles write their partial sums to tile-sized FP32 slices of W.
    const int tile_m = kBM * cg;
    CUtensorMap tmW = tmD;
    if (tail_tiles) {
        st = output_map(h, W, TCG_R_32F, tile_m, kBN, tile_m, (int64_t)tile_m * kBN,
                        tail_tiles * tail.splits, &tmW, c_bufs);
        if (st != TCG_STATUS_SUCCESS)
            return st;
    }

    // One launch of the GEMM kernel: D = alpha * opA * opB + beta * C (with opA2 and opB2,
    // the low words of the two-word split: D = alpha * (opA2 opB + opA opB2 + opA opB) + ...).
    auto gemm_launch = [&](const void *opA, const void *opB, float beta, const void *opA2,
                           const void *opB2) -> tcgStatus_t {
        GemmArgs a;
        std::memset(&a, 0, sizeof a);
        a.m = m; a.n = n; a.k = k; a.batch = batch;
        a.num_m_tiles = (m + kBM * cg - 1) / (kBM * cg);
        a.num_n_tiles = (n + bn - 1) / bn;
        const int es = elem_size(at);
        a.k_row = 128 / es;                           // one 128-byte swizzle row of K
        a.num_k_blocks = (k + kDepth * a.k_row - 1) / (kDepth * a.k_row);
        a.k_splits = plan.splits;
        a.kb_per_split = plan.kb_per_split;
        if (tail_tiles) {
            a.full_units = static_cast<int>(tail.full_tiles);
            a.tail_splits = tail.splits;
            a.tail_kb_per_split = tail.kb_per_split;
            a.total_tiles = a.full_units + static_cast<int>(tail_tiles) * tail.splits;
        } else {
            a.total_tiles = a.num_m_tiles * a.num_n_tiles * batch * plan.splits;
            a.full_units = a.total_tiles;
            a.tail_splits = 1;
            a.tail_kb_per_split = a.num_k_blocks;
        }
        a.group_m = h->group_m > 0 ? h->group_m : 8;
        a.kind = fuse ? (split3 ? kKindTF32x3R : kKindTF32R) : kind;
        if (fuse) {
            const int64_t kp = (p.k + 3) / 4 * 4;
            const bool src_kmajor[2] = {p.transa == TCG_OP_T, p.transb == TCG_OP_N};
            const void *src[2] = {p.A, p.B};
            const int64_t ld_src[2] = {p.lda, p.ldb};
            const int64_t s_src[2] = {p.batched ? p.strideA : 0, p.batched ? p.strideB : 0};
            void *dst[2] = {const_cast<void *>(Aop), const_cast<void *>(Bop)};
            void *dst_lo[2] = {const_cast<void *>(Alo), const_cast<void *>(Blo)};
            const int rows[2] = {m, n};
            const int prow[2] = {kBM * cg, bn};
            const int panels[2] = {cvp.panels_a, cvp.panels_b};
            const int64_t nb[2] = {nba0, nbb0};
            for (int x = 0; x < 2; ++x) {
                a.cv_src[x] = src[x];
                a.cv_dst[x] = dst[x];
                a.cv_dst_lo[x] = dst_lo[x];
                a.cv_ld[x] = ld_src[x];
                a.cv_stride[x] = s_src[x];
                a.cv_dstride[x] = s_src[x] == 0 ? 0 : rows[x] * kp;
                a.cv_kmajor[x] = src_kmajor[x] ? 1 : 0;
                a.cv_rows[x] = rows[x];
                a.cv_panel_rows[x] = prow[x];
                a.cv_panels[x] = panels[x];
                a.cv_subs[x] = (prow[x] / kCvRows) * (kCvChunk / kCvK);
            }
            a.cv_base[0] = 0;
            a.cv_base[1] = static_cast<int>(nb[0] * panels[0] * cvp.chunks);
            a.cv_pbase[0] = 0;
            a.cv_pbase[1] = static_cast<int>(nb[0] * panels[0]);
            a.cv_kp = kp;
            a.cv_kc = kCvChunk;
            a.cv_chunks = cvp.chunks;
            a.cv_kb_per_chunk = kCvChunk / (kDepth * (128 / 4));
            a.cv_items = static_cast<int>(cvp.items);
            a.cv_cnt = cv_cnt;
        }
        // operand format codes: kind::f16 F16 = 0, BF16 = 1; kind::tf32 TF32 = 2;
        // kind::f8f6f4 E4M3 = 0, E5M2 = 1
        const uint32_t fmt = tf32 ? 2u
                                  : (fp8 ? (p.Atype == TCG_R_8F_E5M2 ? 1u : 0u)
                                         : (p.Atype == TCG_R_16BF ? 1u : 0u));
        a.idesc = (1u << 4)                               // D: FP32
                  | (fmt << 7) | (fmt << 10)              // A, B formats
                  | ((a_kmajor ? 0u : 1u) << 15)          // A: 0 = K-major, 1 = M-major
                  | ((b_kmajor ? 0u : 1u) << 16)          // B: 0 = K-major, 1 = N-major
                  | (static_cast<uint32_t>(bn >> 3) << 17)           // N = 256 or 128
                  | (static_cast<uint32_t>((kBM * cg) >> 4) << 24);   // M = 128 or 256
        // Split, the kernel writes the raw FP32 accumulators (alpha 1, beta 0) into the
        // partial-sum slices and the reduction applies alpha and beta.
        a.alpha = splitk ? 1.0f : p.alpha;
        a.beta = splitk ? 0.0f : beta;
        a.c_bufs = a.beta == 0.0f ? 0 : c_bufs;
        a.C = splitk ? static_cast<const void *>(W) : p.C;
        a.D = splitk ? static_cast<void *>(W) : p.C;
        a.ldc = splitk ? ldw : p.ldc;
        a.strideC = splitk ? ldw * p.n : strideC;
        a.err = h->d_err;
        a.wait_limit_ns = h->wait_limit_ns;
        a.fault_inject = h->fault_inject;
        a.clk = h->clk_on ? h->d_clk : nullptr;
        CUtensorMap tmA, tmB;
        bool abc = false, bbc = false;
        tcgStatus_t s2 = operand_map(h, opA, at, a_kmajor, p.m, p.k, lda, sA, p.batch, kBM,
                                     a.k_row, &abc, &a.a_mode, &tmA);
        if (s2 != TCG_STATUS_SUCCESS)
            return s2;
        s2 = operand_map(h, opB, at, b_kmajor, p.n, p.k, ldb, sB, p.batch, bn / cg, a.k_row,
                         &bbc, &a.b_mode, &tmB);
        if (s2 != TCG_STATUS_SUCCESS)
            return s2;
        a.a_bcast = abc ? 1 : 0;
        a.b_bcast = bbc ? 1 : 0;
        // An operand whose rows meet a single tile along the other dimension, and that no
        // other batch entry shares, is read exactly once (e.g. a batch of one-tile
        // products): its loads need not stay in L2.  Measured on GB300, 512 batched
        // 256^3 FP16 products, back-to-back calls: 58.3 -> 51.1 us (C and D then stay in
        // L2); with L2 flushed between calls 59.4 us either way.
        a.a_once = (!abc && a.num_n_tiles == 1) ? 1 : 0;
        a.b_once = (!bbc && a.num_m_tiles == 1) ? 1 : 0;
        CUtensorMap tmA2, tmB2;
        if (opA2) {
            int mode_lo = 0;
            s2 = operand_map(h, opA2, at, a_kmajor, p.m, p.k, lda, sA, p.batch, kBM, a.k_row,
                             &abc, &mode_lo, &tmA2);
            if (s2 == TCG_STATUS_SUCCESS)
                s2 = operand_map(h, opB2, at, b_kmajor, p.n, p.k, ldb, sB, p.batch, bn / cg,
                                 a.k_row, &bbc, &mode_lo, &tmB2);
            if (s2 != TCG_STATUS_SUCCESS)
                return s2;
        }
        const int64_t want = static_cast<int64_t>(a.total_tiles) * cg;
        const int grid = static_cast<int>(want < h->max_ctas[cg] ? want : h->max_ctas[cg]);
        cudaError_t e = launch_gemm(tmA, tmB, tmD, tmW, a,
                                    splitk ? static_cast<int>(kOutF32) : ok, cg, bn, grid,
                                    h->stream, opA2 ? &tmA2 : nullptr, opB2 ? &tmB2 : nullptr);
        h->launches += 1;
        if (e == cudaSuccess && tail_tiles) {
            int64_t blocks = tail_tiles * (kBN / 16);  // 16 columns of a tail tile per block
            const int64_t cap = static_cast<int64_t>(h->num_sms) * 8;
            if (blocks > cap)
                blocks = cap;
            e = launch_tail_reduce(W, static_cast<int>(tail_tiles), tile_m, a,
                                   static_cast<int>(blocks), h->stream);
            h->launches += 1;
        }
        if (e == cudaSuccess && splitk) {
            int64_t blocks = p.n * p.batch;             // one column of D per block
            const int64_t cap = static_cast<int64_t>(h->num_sms) * 8;
            if (blocks > cap)
                blocks = cap;
            e = launch_splitk_reduce(W, ldw, plan.splits, m, n, batch, p.alpha, beta, p.C,
                                     p.ldc, strideC, ok, static_cast<int>(blocks), h->stream);
            h->launches += 1;
        }
        return e == cudaSuccess ? TCG_STATUS_SUCCESS : TCG_STATUS_EXECUTION_FAILED;
    };

    // The split: three products per K slice, the small ones first, accumulated in one FP32
    // accumulator ("NVIDIA Tensor Core混合精度计算原理与应用解析", section 5.1);
    // lo_A * lo_B (<= 2^-22 relative) is dropped.
    return gemm_launch(Aop, Bop, p.beta, split3 ? Alo : nullptr, split3 ? Blo : nullptr);
}


// ---------------------------------------------------------------- host-buffer calls
//
// The same GEMM with A, B and C in host memory: the operands are copied to device
// buffers the handle keeps (same leading dimensions and strides as on the host), the
// product runs on the handle's stream, and D is copied back into C.  The work is cut into
// chunks -- up to kHostPanels column panels of B/C or groups of batch entries, or, for a
// single product of at least 8 waves, a grid of up to 4 x 4 blocks of D -- so that the
// copies of one chunk overlap the product of another (copies in on one stream, copies out
// on another).  Chunk edges fall on tile edges and no chunk splits K (a problem that
// would split its last tiles is run whole): the result is the device call's, bit for bit.

// Elements spanned by a column-major rows x cols matrix with leading dimension ld, and
// by `batch` of them stride elements apart (stride 0: one shared matrix).
int64_t span(int64_t rows, int64_t cols, int64_t ld, int64_t batch, int64_t stride)
{
    if (rows == 0 || cols == 0 || batch == 0)
        return 0;
    const int64_t one = (cols - 1) * ld + rows;
    return stride == 0 ? one : (batch - 1) * stride + one;
}

tcgStatus_t stage_buffer(tcgContext *h, int i, size_t bytes, void **out)
{
    if (h->stage_bytes[i] < bytes) {
        if (h->stage_buf[i]) {
            cudaDeviceSynchronize();
            cudaFree(h->stage_buf[i]);
            h->stage_buf[i] = nullptr;
            h->stage_bytes[i] = 0;
        }
        if (cudaMalloc(&h->stage_buf[i], bytes ? bytes : 16) != cudaSuccess) {
            cudaGetLastError();
            h->stage_buf[i] = nullptr;
            return TCG_STATUS_ALLOC_FAILED;
        }
        h->stage_bytes[i] = bytes;
    }
    *out = h->stage_buf[i];
    return TCG_STATUS_SUCCESS;
}

tcgStatus_t host_streams(tcgContext *h)
{
    if (!h->h2d && cudaStreamCreateWithFlags(&h->h2d, cudaStreamNonBlocking) != cudaSuccess)
        return TCG_STATUS_EXECUTION_FAILED;
    if (!h->d2h && cudaStreamCreateWithFlags(&h->d2h, cudaStreamNonBlocking) != cudaSuccess)
        return TCG_STATUS_EXECUTION_FAILED;
    for (int i = 0; i < kHostChunks; ++i) {
        if (!h->ev_in[i] && cudaEventCreateWithFlags(&h->ev_in[i], cudaEventDisableTiming) != cudaSuccess)
            return TCG_STATUS_EXECUTION_FAILED;
        if (!h->ev_out[i] && cudaEventCreateWithFlags(&h->ev_out[i], cudaEventDisableTiming) != cudaSuccess)
            return TCG_STATUS_EXECUTION_FAILED;
    }
    return TCG_STATUS_SUCCESS;
}

tcgStatus_t run_host(tcgContext *h, const Problem &hp)
{
    // Host memory needs no particular alignment (the device copies get cudaMalloc's): check
    // the arguments with stand-in aligned addresses where pointers were given.
    Problem cp = hp;
    static const uint4 stand_in = {0, 0, 0, 0};
    if (cp.A) cp.A = &stand_in;
    if (cp.B) cp.B = &stand_in;
    if (cp.C) cp.C = const_cast<uint4 *>(&stand_in);
    tcgStatus_t st = check_args(cp);
    if (st != TCG_STATUS_SUCCESS)
        return st;
    if (hp.m == 0 || hp.n == 0 || hp.batch == 0)
        return TCG_STATUS_SUCCESS;
    st = bind_device(h);
    if (st != TCG_STATUS_SUCCESS)
        return st;
    st = host_streams(h);
    if (st != TCG_STATUS_SUCCESS) {
        cudaGetLastError();
        return st;
    }
    h->used = true;
    const bool product = hp.k > 0 && hp.alpha != 0.0f;
    const bool read_c = hp.beta != 0.0f;
    const int64_t esa = elem_size(hp.Atype), esc = elem_size(hp.Ctype);
    const int64_t a_rows = hp.transa == TCG_OP_N ? hp.m : hp.k;
    const int64_t a_cols = hp.transa == TCG_OP_N ? hp.k : hp.m;
    const int64_t b_rows = hp.transb == TCG_OP_N ? hp.k : hp.n;
    const int64_t b_cols = hp.transb == TCG_OP_N ? hp.n : hp.k;
    const int64_t sA = hp.batched ? hp.strideA : 0, sB = hp.batched ? hp.strideB : 0;
    const int64_t sC = hp.batched ? hp.strideC : 0;
    const int64_t nA = product ? span(a_rows, a_cols, hp.lda, hp.batch, sA) : 0;
    const int64_t nB = product ? span(b_rows, b_cols, hp.ldb, hp.batch, sB) : 0;
    const int64_t nC = span(hp.m, hp.n, hp.ldc, hp.batch, sC);
    void *dA = nullptr, *dB = nullptr, *dC = nullptr;
    if ((st = stage_buffer(h, 0, (size_t)(nA * esa), &dA)) != TCG_STATUS_SUCCESS ||
        (st = stage_buffer(h, 1, (size_t)(nB * esa), &dB)) != TCG_STATUS_SUCCESS ||
        (st = stage_buffer(h, 2, (size_t)(nC * esc), &dC)) != TCG_STATUS_SUCCESS)
        return st;

    // Chunks: column panels (one matrix) or batch groups, each at least one wave of tiles.
    if (h->max_ctas[h->cta_group] == 0)
        h->max_ctas[h->cta_group] = gemm_max_resident_ctas(h->cta_group, h->num_sms);
    const int64_t clusters = h->max_ctas[h->cta_group] / h->cta_group;
    const int64_t tile_m = kBM * h->cta_group;
    const int64_t m_tiles = (hp.m + tile_m - 1) / tile_m, n_tiles = (hp.n + kBN - 1) / kBN;
    const int64_t units = hp.batched ? hp.batch : n_tiles;        // what chunks split
    const int64_t per_unit = hp.batched ? m_tiles * n_tiles : m_tiles;
    int64_t chunks = clusters > 0 ? per_unit * units / clusters : 1;
    chunks = chunks < 1 ? 1 : (chunks > kHostPanels ? kHostPanels : chunks);
    {   // a problem whose last tiles are K-split is run whole (chunks would tile differently)
        const bool tf32c = hp.compute != TCG_COMPUTE_32F;
        const int es_k = tf32c ? 4 : elem_size(hp.Atype);
        const SplitPlan sp = plan_for(h, hp.m, hp.n, hp.k, hp.batch, es_k, h->cta_group);
        if (tail_for(h, hp.m, hp.n, hp.k, hp.batch, es_k, h->cta_group,
                     hp.Ctype == TCG_R_32F, sp).splits > 1)
            chunks = 1;
    }
    if (chunks > units)
        chunks = units;
    const int64_t per_chunk = (units + chunks - 1) / chunks;      // units per chunk
    chunks = (units + per_chunk - 1) / per_chunk;
    // A problem of several waves is never split along K (see split_plan); its chunks, some
    // smaller than a wave, must not be either.  A forced split applies to every chunk alike.
    const int saved_split = h->split_k;
    if (chunks > 1 && saved_split == 0)
        h->split_k = 1;
    struct Restore {
        tcgContext *h;
        int v;
        ~Restore() { h->split_k = v; }
    } restore{h, saved_split};

    auto fail = [&]() {
        cudaGetLastError();
        cudaStreamSynchronize(h->h2d);
        cudaStreamSynchronize(h->d2h);
        cudaStreamSynchronize(h->stream);
        cudaGetLastError();
        return TCG_STATUS_EXECUTION_FAILED;
    };
    auto h2d = [&](void *dst, const void *src, int64_t bytes) {
        return bytes <= 0 ||
               cudaMemcpyAsync(dst, src, (size_t)bytes, cudaMemcpyHostToDevice, h->h2d) == cudaSuccess;
    };
    const char *A = static_cast<const char *>(hp.A);
    const char *B = static_cast<const char *>(hp.B);
    char *C = static_cast<char *>(hp.C);
    char *dAc = static_cast<char *>(dA), *dBc = static_cast<char *>(dB), *dCc = static_cast<char *>(dC);
    // Work on the handle's stream issued before this call must not see the staging
    // buffers change under it: copies start after it.
    if (cudaEventRecord(h->ev_out[0], h->stream) != cudaSuccess ||
        cudaStreamWaitEvent(h->h2d, h->ev_out[0], 0) != cudaSuccess)
        return fail();
    // A large single product (at least 8 waves of tiles) goes as a grid of up to 4 x 4
    // blocks of D.  Block (i, j) needs block row i of op(A) and block column j of op(B);
    // each goes in once, in the order of first use, so that D's blocks start going out
    // after the first row block of A and column block of B have arrived instead of after
    // all of A, and the two directions of the host link stay busy together.  Block edges
    // fall on tile edges, so every tile is accumulated exactly as in the whole call.
    if (!hp.batched && product && chunks > 1 && m_tiles * n_tiles >= 8 * clusters) {
        const int64_t mt_per = (m_tiles + 3) / 4, nt_per = (n_tiles + 3) / 4;
        const int64_t mc = (m_tiles + mt_per - 1) / mt_per, nc = (n_tiles + nt_per - 1) / nt_per;
        auto copy_a = [&](int64_t i0, int64_t i1) {
            if (hp.transa == TCG_OP_N)                 // rows i0..i1 of an m x k matrix
                return cudaMemcpy2DAsync(dAc + i0 * esa, (size_t)(hp.lda * esa), A + i0 * esa,
                                         (size_t)(hp.lda * esa), (size_t)((i1 - i0) * esa),
                                         (size_t)hp.k, cudaMemcpyHostToDevice, h->h2d) == cudaSuccess;
            const int64_t off = i0 * hp.lda;           // columns i0..i1 of a k x m matrix
            return h2d(dAc + off * esa, A + off * esa, span(hp.k, i1 - i0, hp.lda, 1, 0) * esa);
        };
        auto copy_b = [&](int64_t j0, int64_t j1) {
            if (hp.transb == TCG_OP_N) {               // columns j0..j1 of a k x n matrix
                const int64_t off = j0 * hp.ldb;
                return h2d(dBc + off * esa, B + off * esa, span(hp.k, j1 - j0, hp.ldb, 1, 0) * esa);
            }                                          // rows j0..j1 of an n x k matrix
            return cudaMemcpy2DAsync(dBc + j0 * esa, (size_t)(hp.ldb * esa), B + j0 * esa,
                                     (size_t)(hp.ldb * esa), (size_t)((j1 - j0) * esa),
                                     (size_t)hp.k, cudaMemcpyHostToDevice, h->h2d) == cudaSuccess;
        };
        // rows i0..i1 of columns j0..j1 of C / D, in either direction
        auto copy_block = [&](char *dst, const char *src, int64_t i0, int64_t i1, int64_t j0,
                              int64_t j1, cudaMemcpyKind kind, cudaStream_t s) {
            const int64_t off = (i0 + j0 * hp.ldc) * esc;
            return cudaMemcpy2DAsync(dst + off, (size_t)(hp.ldc * esc), src + off,
                                     (size_t)(hp.ldc * esc), (size_t)((i1 - i0) * esc),
                                     (size_t)(j1 - j0), kind, s) == cudaSuccess;
        };
        // Blocks in growing squares (square q: the blocks with max(i, j) = q, first (q, 0..q-1)
        // then (0..q, q)), so that each new block row of A and column of B is followed by
        // the blocks it completes and the copies out keep pace with the copies in.
        int64_t order_i[kHostChunks], order_j[kHostChunks], nblocks = 0;
        for (int64_t q = 0; q < (mc > nc ? mc : nc); ++q)
            for (int64_t r = 0; r < 2 * q + 1; ++r) {
                const int64_t i = r < q ? q : r - q, j = r < q ? r : q;
                if (i < mc && j < nc) {
                    order_i[nblocks] = i;
                    order_j[nblocks] = j;
                    ++nblocks;
                }
            }
        bool a_in[4] = {false, false, false, false}, b_in[4] = {false, false, false, false};
        for (int64_t c = 0; c < nblocks; ++c) {
            const int64_t i = order_i[c], j = order_j[c];
            const int64_t i0 = i * mt_per * tile_m;
            const int64_t i1 = (i + 1) * mt_per * tile_m < hp.m ? (i + 1) * mt_per * tile_m : hp.m;
            const int64_t j0 = j * nt_per * kBN;
            const int64_t j1 = (j + 1) * nt_per * kBN < hp.n ? (j + 1) * nt_per * kBN : hp.n;
            if ((!a_in[i] && !copy_a(i0, i1)) || (!b_in[j] && !copy_b(j0, j1)) ||
                (read_c && !copy_block(dCc, C, i0, i1, j0, j1, cudaMemcpyHostToDevice, h->h2d)))
                return fail();
            a_in[i] = b_in[j] = true;
            if (cudaEventRecord(h->ev_in[c], h->h2d) != cudaSuccess ||
                cudaStreamWaitEvent(h->stream, h->ev_in[c], 0) != cudaSuccess)
                return fail();
            Problem dp = hp;
            dp.staged = true;
            dp.m = i1 - i0;
            dp.n = j1 - j0;
            dp.A = hp.transa == TCG_OP_N ? dAc + i0 * esa : dAc + i0 * hp.lda * esa;
            dp.B = hp.transb == TCG_OP_N ? dBc + j0 * hp.ldb * esa : dBc + j0 * esa;
            dp.C = dCc + (i0 + j0 * hp.ldc) * esc;
            st = run(h, dp);
            if (st != TCG_STATUS_SUCCESS) {
                fail();
                return st;
            }
            if (cudaEventRecord(h->ev_out[c], h->stream) != cudaSuccess ||
                cudaStreamWaitEvent(h->d2h, h->ev_out[c], 0) != cudaSuccess ||
                !copy_block(C, dCc, i0, i1, j0, j1, cudaMemcpyDeviceToHost, h->d2h))
                return fail();
        }
        if (cudaStreamSynchronize(h->d2h) != cudaSuccess || cudaStreamSynchronize(h->h2d) != cudaSuccess)
            return fail();
        return TCG_STATUS_SUCCESS;
    }
    // A whole (or, batched, per group below when it has a stride).
    const bool a_per_group = hp.batched && sA != 0;
    if (product && !a_per_group && !h2d(dAc, A, nA * esa))
        return fail();
    for (int64_t c = 0; c < chunks; ++c) {
        const int64_t u0 = c * per_chunk, u1 = u0 + per_chunk < units ? u0 + per_chunk : units;
        Problem dp = hp;
        dp.staged = true;
        dp.A = dA;
        dp.B = dB;
        dp.C = dC;
        // element ranges of this chunk (in the host/device layouts, which are the same)
        int64_t c_off, c_len;
        if (hp.batched) {
            const int64_t b0 = u0, b1 = u1;
            dp.batch = b1 - b0;
            if (product) {
                if (a_per_group) {
                    const int64_t off = b0 * sA, len = span(a_rows, a_cols, hp.lda, b1 - b0, sA);
                    if (!h2d(dAc + off * esa, A + off * esa, len * esa))
                        return fail();
                    dp.A = dAc + off * esa;
                }
                if (sB != 0) {
                    const int64_t off = b0 * sB, len = span(b_rows, b_cols, hp.ldb, b1 - b0, sB);
                    if (!h2d(dBc + off * esa, B + off * esa, len * esa))
                        return fail();
                    dp.B = dBc + off * esa;
                } else if (c == 0 && !h2d(dBc, B, nB * esa)) {
                    return fail();
                }
            }
            c_off = b0 * sC;
            c_len = span(hp.m, hp.n, hp.ldc, b1 - b0, sC);
            dp.C = dCc + c_off * esc;
        } else {
            const int64_t j0 = u0 * kBN, j1 = u1 * kBN < hp.n ? u1 * kBN : hp.n;
            dp.n = j1 - j0;
            if (product) {
                if (hp.transb == TCG_OP_N) {           // columns j0..j1 of a k x n matrix
                    const int64_t off = j0 * hp.ldb, len = span(hp.k, j1 - j0, hp.ldb, 1, 0);
                    if (!h2d(dBc + off * esa, B + off * esa, len * esa))
                        return fail();
                    dp.B = dBc + off * esa;
                } else {                               // rows j0..j1 of an n x k matrix
                    if (cudaMemcpy2DAsync(dBc + j0 * esa, (size_t)(hp.ldb * esa), B + j0 * esa,
                                          (size_t)(hp.ldb * esa), (size_t)((j1 - j0) * esa),
                                          (size_t)hp.k, cudaMemcpyHostToDevice, h->h2d) != cudaSuccess)
                        return fail();
                    dp.B = dBc + j0 * esa;
                }
            }
            c_off = j0 * hp.ldc;
            c_len = span(hp.m, j1 - j0, hp.ldc, 1, 0);
            dp.C = dCc + c_off * esc;
        }
        if (read_c && !h2d(dCc + c_off * esc, C + c_off * esc, c_len * esc))
            return fail();
        if (cudaEventRecord(h->ev_in[c], h->h2d) != cudaSuccess ||
            cudaStreamWaitEvent(h->stream, h->ev_in[c], 0) != cudaSuccess)
            return fail();
        st = run(h, dp);
        if (st != TCG_STATUS_SUCCESS) {
            fail();
            return st;
        }
        if (cudaEventRecord(h->ev_out[c], h->stream) != cudaSuccess ||
            cudaStreamWaitEvent(h->d2h, h->ev_out[c], 0) != cudaSuccess)
            return fail();
        // D back into C, leaving the ldc padding and the gaps between batch entries alone.
        cudaError_t e = cudaSuccess;
        const int64_t cols = hp.batched ? hp.n : dp.n;
        const int64_t nb = hp.batched ? dp.batch : 1;
        if (hp.ldc == hp.m && (nb == 1 || sC == hp.m * hp.n)) {
            e = cudaMemcpyAsync(C + c_off * esc, dCc + c_off * esc, (size_t)(hp.m * cols * nb * esc),
                                cudaMemcpyDeviceToHost, h->d2h);
        } else if (hp.ldc == hp.m) {
            e = cudaMemcpy2DAsync(C + c_off * esc, (size_t)(sC * esc), dCc + c_off * esc,
                                  (size_t)(sC * esc), (size_t)(hp.m * cols * esc), (size_t)nb,
                                  cudaMemcpyDeviceToHost, h->d2h);
        } else {
            for (int64_t b = 0; b < nb && e == cudaSuccess; ++b)
                e = cudaMemcpy2DAsync(C + (c_off + b * sC) * esc, (size_t)(hp.ldc * esc),
                                      dCc + (c_off + b * sC) * esc, (size_t)(hp.ldc * esc),
                                      (size_t)(hp.m * esc), (size_t)cols, cudaMemcpyDeviceToHost,
                                      h->d2h);
        }
        if (e != cudaSuccess)
            return fail();
    }
    if (cudaStreamSynchronize(h->d2h) != cudaSuccess || cudaStreamSynchronize(h->h2d) != cudaSuccess)
        return fail();
    return TCG_STATUS_SUCCESS;
}

}  // namespace

extern "C" {

tcgStatus_t tcg_create(tcgHandle_t *h)
{
    if (!h)
        return TCG_STATUS_INVALID_VALUE;
    tcgContext *c = new (std::nothrow) tcgContext();
    if (!c)
        return TCG_STATUS_ALLOC_FAILED;
    *h = c;
    return TCG_STATUS_SUCCESS;
}

tcgStatus_t tcg_destroy(tcgHandle_t h)
{
    if (!h)
        return TCG_STATUS_INVALID_VALUE;
    // Drain every stream that may still use the handle's memory before freeing it.
    if (h->used)
        cudaStreamSynchronize(h->stream);
    if (h->h2d)
        cudaStreamSynchronize(h->h2d);
    if (h->d2h)
        cudaStreamSynchronize(h->d2h);
    if (h->d_err)
        cudaFree(h->d_err);
    if (h->d_clk)
        cudaFree(h->d_clk);
    if (h->ws_own)
        cudaFree(h->ws_own);
    for (int i = 0; i < 3; ++i)
        if (h->stage_buf[i])
            cudaFree(h->stage_buf[i]);
    if (h->h2d)
        cudaStreamDestroy(h->h2d);
    if (h->d2h)
        cudaStreamDestroy(h->d2h);
    for (int i = 0; i < kHostChunks; ++i) {
        if (h->ev_in[i])
            cudaEventDestroy(h->ev_in[i]);
        if (h->ev_out[i])
            cudaEventDestroy(h->ev_out[i]);
    }
    delete h;
    return TCG_STATUS_SUCCESS;
}

tcgStatus_t tcg_set_stream(tcgHandle_t h, void *stream)
{
    if (!h)
        return TCG_STATUS_INVALID_VALUE;
    h->stream = static_cast<cudaStream_t>(stream);
    return TCG_STATUS_SUCCESS;
}

tcgStatus_t tcg_set_workspace(tcgHandle_t h, void *ptr, size_t bytes)
{
    if (!h || (bytes > 0 && !ptr) || (reinterpret_cast<uintptr_t>(ptr) & 255u))
        return TCG_STATUS_INVALID_VALUE;
    h->ws_user = bytes ? ptr : nullptr;
    h->ws_user_bytes = bytes;
    return TCG_STATUS_SUCCESS;
}

tcgStatus_t tcg_gemm_workspace_size(tcgOp_t transa, tcgOp_t transb, int64_t m, int64_t n,
                                    int64_t k, tcgDataType_t Atype, tcgComputeType_t compute,
                                    int64_t batch_count, size_t *bytes)
{
    (void)transa;
    (void)transb;
    if (!bytes || m < 0 || n < 0 || k < 0 || batch_count < 0 || !valid_type(Atype))
        return TCG_STATUS_INVALID_VALUE;
    *bytes = 0;
    if (Atype == TCG_R_32F && k > 0) {
        if (compute == TCG_COMPUTE_32F_FAST_TF32)   // copies + in-kernel rounding counters
            *bytes = tf32_ws_bytes(m, n, k, batch_count) +
                     cv_ws_bytes(cv_plan(m, n, k, batch_count, batch_count, kBM, kBNNarrow));
        else if (compute == TCG_COMPUTE_32F_3XTF32)
            *bytes = 2 * tf32_ws_bytes(m, n, k, batch_count) +
                     cv_ws_bytes(cv_plan(m, n, k, batch_count, batch_count, kBM, kBNNarrow));
    }
    // Split-K partial sums, as a handle with default options would split on the current
    // device (its SM count; at most kMaxSplits slices).
    if (k > 0 && m > 0 && n > 0 && batch_count > 0) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();          // no device: no GEMM can run, nothing to split
            return TCG_STATUS_SUCCESS;
        }
        const int es = Atype == TCG_R_32F ? 4 : elem_size(Atype);
        const int64_t k_block = static_cast<int64_t>(kDepth) * (128 / es);
        const int nkb = static_cast<int>((k + k_block - 1) / k_block);
        const int64_t tiles = ((m + 2 * kBM - 1) / (2 * kBM)) * ((n + kBN - 1) / kBN) * batch_count;
        const SplitPlan pl = split_plan(tiles, nkb, sms / 2, 0);
        if (pl.splits > 1) {
            *bytes += splitk_ws_bytes(m, n, batch_count, pl.splits);
        } else {        // tail split of an FP32-output call
            const TailPlan tp = tail_plan(tiles, nkb, sms / 2, nkb * 512.0 * kDepth / 1.8e3,
                                          4.0 * 2 * kBM * kBN);
            if (tp.splits > 1)
                *bytes += (size_t)((tiles - tp.full_tiles) * tp.splits) * (size_t)(2 * kBM * kBN) * 4;
        }
    }
    return TCG_STATUS_SUCCESS;
}

tcgStatus_t tcg_gemm_ex(tcgHandle_t h, tcgOp_t transa, tcgOp_t transb, int64_t m, int64_t n,
                        int64_t k, float alpha, const void *A, tcgDataType_t Atype,
                        int64_t lda, const void *B, tcgDataType_t Btype, int64_t ldb,
                        float beta, void *C, tcgDataType_t Ctype, int64_t ldc,
                        tcgComputeType_t compute)
{
    if (!h)
        return TCG_STATUS_INVALID_VALUE;
    Problem p{transa, transb, m, n, k, alpha, beta, A, Atype, lda, 0, B, Btype, ldb, 0,
              C, Ctype, ldc, 0, 1, compute, false};
    return run(h, p);
}

tcgStatus_t tcg_gemm_strided_batched(tcgHandle_t h, tcgOp_t transa, tcgOp_t transb,
                                     int64_t m, int64_t n, int64_t k, float alpha,
                                     const void *A, tcgDataType_t Atype, int64_t lda,
                                     int64_t strideA, const void *B, tcgDataType_t Btype,
                                     int64_t ldb, int64_t strideB, float beta, void *C,
                                     tcgDataType_t Ctype, int64_t ldc, int64_t strideC,
                                     int64_t batch_count, tcgComputeType_t compute)
{
    if (!h)
        return TCG_STATUS_INVALID_VALUE;
    Problem p{transa, transb, m, n, k, alpha, beta, A, Atype, lda, strideA, B, Btype, ldb,
              strideB, C, Ctype, ldc, strideC, batch_count, compute, true};
    return run(h, p);
}

tcgStatus_t tcg_gemm_ex_host(tcgHandle_t h, tcgOp_t transa, tcgOp_t transb, int64_t m, int64_t n,
                             int64_t k, float alpha, const void *A, tcgDataType_t Atype,
                             int64_t lda, const void *B, tcgDataType_t Btype, int64_t ldb,
                             float beta, void *C, tcgDataType_t Ctype, int64_t ldc,
                             tcgComputeType_t compute)
{
    if (!h)
        return TCG_STATUS_INVALID_VALUE;
    Problem p{transa, transb, m, n, k, alpha, beta, A, Atype, lda, 0, B, Btype, ldb, 0,
              C, Ctype, ldc, 0, 1, compute, false};
    return run_host(h, p);
}

tcgStatus_t tcg_gemm_strided_batched_host(tcgHandle_t h, tcgOp_t transa, tcgOp_t transb,
                                          int64_t m, int64_t n, int64_t k, float alpha,
                                          const void *A, tcgDataType_t Atype, int64_t lda,
                                          int64_t strideA, const void *B, tcgDataType_t Btype,
                                          int64_t ldb, int64_t strideB, float beta, void *C,
                                          tcgDataType_t Ctype, int64_t ldc, int64_t strideC,
                                          int64_t batch_count, tcgComputeType_t compute)
{
    if (!h)
        return TCG_STATUS_INVALID_VALUE;
    Problem p{transa, transb, m, n, k, alpha, beta, A, Atype, lda, strideA, B, Btype, ldb,
              strideB, C, Ctype, ldc, strideC, batch_count, compute, true};
    return run_host(h, p);
}

tcgStatus_t tcg_get_device_error(tcgHandle_t h)
{
    if (!h)
        return TCG_STATUS_INVALID_VALUE;
    if (!h->d_err)
        return TCG_STATUS_SUCCESS;
    uint32_t bits = 0;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess ||
        cudaMemcpy(&bits, h->d_err, sizeof bits, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(h->d_err, 0, sizeof(uint32_t)) != cudaSuccess) {
        cudaGetLastError();
        return TCG_STATUS_EXECUTION_FAILED;
    }
    h->last_err_bits = bits;
    return bits ? TCG_STATUS_TIMEOUT : TCG_STATUS_SUCCESS;
}

uint32_t tcg_last_device_error_bits(tcgHandle_t h) { return h ? h->last_err_bits : 0u; }

const char *tcg_status_string(tcgStatus_t s)
{
    switch (s) {
    case TCG_STATUS_SUCCESS: return "TCG_STATUS_SUCCESS";
    case TCG_STATUS_NOT_INITIALIZED: return "TCG_STATUS_NOT_INITIALIZED";
    case TCG_STATUS_INVALID_VALUE: return "TCG_STATUS_INVALID_VALUE";
    case TCG_STATUS_NOT_SUPPORTED: return "TCG_STATUS_NOT_SUPPORTED";
    case TCG_STATUS_ARCH_MISMATCH: return "TCG_STATUS_ARCH_MISMATCH";
    case TCG_STATUS_EXECUTION_FAILED: return "TCG_STATUS_EXECUTION_FAILED";
    case TCG_STATUS_TIMEOUT: return "TCG_STATUS_TIMEOUT";
    case TCG_STATUS_ALLOC_FAILED: return "TCG_STATUS_ALLOC_FAILED";
    }
    return "TCG_STATUS_UNKNOWN";
}

tcgStatus_t tcg_set_debug(tcgHandle_t h, uint64_t wait_limit_ns, int fault_inject)
{
    if (!h)
        return TCG_STATUS_INVALID_VALUE;
    h->wait_limit_ns = wait_limit_ns ? wait_limit_ns : kDefaultWaitNs;
    h->fault_inject = fault_inject ? 1 : 0;
    return TCG_STATUS_SUCCESS;
}

uint64_t tcg_launch_count(tcgHandle_t h) { return h ? h->launches : 0; }

tcgStatus_t tcg_set_clock_probe(tcgHandle_t h, int on)
{
    if (!h)
        return TCG_STATUS_INVALID_VALUE;
    if (!on) {
        h->clk_on = false;
        return TCG_STATUS_SUCCESS;
    }
    tcgStatus_t st = bind_device(h);
    if (st != TCG_STATUS_SUCCESS)
        return st;
    if (!h->d_clk) {
        if (cudaMalloc(&h->d_clk, 2 * sizeof(unsigned long long)) != cudaSuccess) {
            cudaGetLastError();
            h->d_clk = nullptr;
            return TCG_STATUS_ALLOC_FAILED;
        }
    }
    if (cudaMemsetAsync(h->d_clk, 0, 2 * sizeof(unsigned long long), h->stream) != cudaSuccess) {
        cudaGetLastError();
        return TCG_STATUS_EXECUTION_FAILED;
    }
    h->clk_on = true;
    return TCG_STATUS_SUCCESS;
}

tcgStatus_t tcg_read_clock_probe(tcgHandle_t h, uint64_t *sm_cycles, uint64_t *ns)
{
    if (!h || !sm_cycles || !ns)
        return TCG_STATUS_INVALID_VALUE;
    *sm_cycles = *ns = 0;
    if (!h->d_clk)
        return TCG_STATUS_SUCCESS;
    unsigned long long v[2] = {0, 0};
    if (cudaStreamSynchronize(h->stream) != cudaSuccess ||
        cudaMemcpy(v, h->d_clk, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return TCG_STATUS_EXECUTION_FAILED;
    }
    *sm_cycles = v[0];
    *ns = v[1];
    return TCG_STATUS_SUCCESS;
}

tcgStatus_t tcg_set_kernel_options(tcgHandle_t h, int cta_group, int group_m)
{
    if (!h || cta_group < 0 || cta_group > 2 || group_m < 0 || group_m > 1024)
        return TCG_STATUS_INVALID_VALUE;
    h->cta_group = cta_group ? cta_group : 2;
    h->group_m = group_m;
    return TCG_STATUS_SUCCESS;
}

tcgStatus_t tcg_set_split_k(tcgHandle_t h, int splits)
{
    if (!h || splits < 0 || splits > kMaxSplits)
        return TCG_STATUS_INVALID_VALUE;
    h->split_k = splits;
    return TCG_STATUS_SUCCESS;
}

tcgStatus_t tcg_set_tile_n(tcgHandle_t h, int tile_n)
{
    if (!h || (tile_n != 0 && tile_n != kBN && tile_n != kBNNarrow))
        return TCG_STATUS_INVALID_VALUE;
    h->tile_n = tile_n;
    return TCG_STATUS_SUCCESS;
}

tcgStatus_t tcg_set_tf32_rounding(tcgHandle_t h, int mode)
{
    if (!h || mode < 0 || mode > 2)
        return TCG_STATUS_INVALID_VALUE;
    h->tf32_round = mode;
    return TCG_STATUS_SUCCESS;
}

tcgStatus_t tcg_split_k_plan(int64_t tiles, int num_k_blocks, int clusters, int forced,
                             int *splits, int *kb_per_split)
{
    if (!splits || !kb_per_split || tiles < 0 || num_k_blocks < 0 || clusters < 0 ||
        forced < 0 || forced > kMaxSplits)
        return TCG_STATUS_INVALID_VALUE;
    const SplitPlan pl = split_plan(tiles, num_k_blocks, clusters, forced);
    *splits = pl.splits;
    *kb_per_split = pl.kb_per_split;
    return TCG_STATUS_SUCCESS;
}

tcgStatus_t tcg_tail_split_plan(int64_t tiles, int num_k_blocks, int clusters, double tile_us,
                                double tile_bytes, int64_t *full_tiles, int *splits,
                                int *kb_per_split)
{
    if (!full_tiles || !splits || !kb_per_split || tiles < 0 || num_k_blocks < 0 || clusters < 0)
        return TCG_STATUS_INVALID_VALUE;
    const TailPlan pl = tail_plan(tiles, num_k_blocks, clusters, tile_us, tile_bytes);
    *full_tiles = pl.full_tiles;
    *splits = pl.splits;
    *kb_per_split = pl.kb_per_split;
    return TCG_STATUS_SUCCESS;
}

tcgStatus_t tcg_gemm_tile_plan(tcgHandle_t h, int64_t m, int64_t n, int64_t k,
                               tcgDataType_t Atype, tcgComputeType_t compute, tcgDataType_t Ctype,
                               int64_t batch_count, int64_t max_tiles, int *tile_m, int *tile_n,
                               int *splits, int64_t *k_per_split)
{
    if (!h || !tile_m || !tile_n || m < 0 || n < 0 || k < 0 || batch_count < 0 ||
        !valid_type(Atype) || !valid_type(Ctype))
        return TCG_STATUS_INVALID_VALUE;
    tcgStatus_t st = bind_device(h);
    if (st != TCG_STATUS_SUCCESS)
        return st;
    const int cg = h->cta_group;
    const bool tf32 = compute == TCG_COMPUTE_32F_FAST_TF32 || compute == TCG_COMPUTE_32F_3XTF32;
    const int es = tf32 ? 4 : elem_size(Atype);
    const bool split3 = compute == TCG_COMPUTE_32F_3XTF32;
    const int kind = split3 ? kKindTF32x3
                            : (tf32 ? kKindTF32 : (is_fp8(Atype) ? kKindF8 : kKindF16));
    const int bn = k > 0 ? tile_n_for(h, m, n, k, batch_count, es, cg, kind) : kBN;
    *tile_m = kBM * cg;
    *tile_n = bn;
    const int64_t k_row = 128 / es, k_block = kDepth * k_row;
    GemmArgs a;
    std::memset(&a, 0, sizeof a);
    a.num_m_tiles = static_cast<int>((m + kBM * cg - 1) / (kBM * cg));
    a.num_n_tiles = static_cast<int>((n + bn - 1) / bn);
    a.group_m = h->group_m > 0 ? h->group_m : 8;
    const int64_t tiles = static_cast<int64_t>(a.num_m_tiles) * a.num_n_tiles * batch_count;
    if (max_tiles < tiles || (tiles > 0 && (!splits || !k_per_split)))
        return TCG_STATUS_INVALID_VALUE;
    if (tiles == 0 || k == 0)
        return TCG_STATUS_SUCCESS;
    const SplitPlan sp = plan_for(h, m, n, k, batch_count, es, cg, bn);
    const TailPlan tp = tail_for(h, m, n, k, batch_count, es, cg, Ctype == TCG_R_32F, sp, bn,
                                 split3 ? 3.0 : 1.0);
    // tiles in raster order -> (b, mt, nt); entry b * mt_count * nt_count + mt * nt_count + nt
    for (int64_t t = 0; t < tiles; ++t) {
        int b, mt, nt;
        raster(a, static_cast<int>(t), b, mt, nt);
        const int64_t e = (static_cast<int64_t>(b) * a.num_m_tiles + mt) * a.num_n_tiles + nt;
        if (tp.splits > 1 && t >= tp.full_tiles) {
            splits[e] = tp.splits;
            k_per_split[e] = static_cast<int64_t>(tp.kb_per_split) * k_block;
        } else {
            splits[e] = sp.splits;
            k_per_split[e] = sp.splits > 1 ? static_cast<int64_t>(sp.kb_per_split) * k_block : k;
        }
    }
    return TCG_STATUS_SUCCESS;
}

tcgStatus_t tcg_gemm_split_k(tcgHandle_t h, int64_t m, int64_t n, int64_t k,
                             tcgDataType_t Atype, tcgComputeType_t compute, int64_t batch_count,
                             int *splits, int64_t *k_per_split)
{
    if (!h || !splits || !k_per_split || m < 0 || n < 0 || k < 0 || batch_count < 0 ||
        !valid_type(Atype))
        return TCG_STATUS_INVALID_VALUE;
    tcgStatus_t st = bind_device(h);
    if (st != TCG_STATUS_SUCCESS)
        return st;
    const bool tf32 = compute == TCG_COMPUTE_32F_FAST_TF32 || compute == TCG_COMPUTE_32F_3XTF32;
    const int es = tf32 ? 4 : elem_size(Atype);
    const SplitPlan pl = plan_for(h, m, n, k, batch_count, es, h->cta_group);
    *splits = pl.splits;
    *k_per_split = static_cast<int64_t>(pl.kb_per_split) * kDepth * (128 / es);
    return TCG_STATUS_SUCCESS;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free TF32 GEMM (tcg_gemm_tf32_noalloc).
//
// Some callers cannot allocate device memory at the moment they multiply: a
// latency-critical loop cannot afford cudaMalloc/cudaFree (they synchronise the
// device and take unbounded time), and a process whose device memory is owned by
// another allocator (a framework's caching pool, a fixed memory budget) must not
// make raw allocations behind that allocator's back.  The TF32 path needs scratch
// memory for its rounded, K-major operand copies, so this entry point keeps that
// scratch in a fixed array compiled into the library instead of a workspace.
//
// The array is a file-scope __device__ object: every GPU that loads the library
// holds it (kNoAllocScratchBytes) until the process exits.  Host code must not
// use its name as a pointer (on the host it only stands in for the symbol); the
// device address is looked up once per device and context with
// cudaGetSymbolAddress: a cudaDeviceReset ends the context, and with it the
// addresses, so a call made in a new context looks them up again.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;   // 32 MiB

__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];
__device__ __align__(256) uint32_t g_noalloc_err;

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

struct NoAllocDevice {
    bool ready = false;
    unsigned long long ctx_id = 0;   // the context the addresses below belong to
    void *scratch = nullptr;     // device address of g_noalloc_scratch
    uint32_t *err = nullptr;     // device address of g_noalloc_err
    EncodeTiledFn encode = nullptr;
    int num_sms = 0;
    int max_ctas = 0;
};

constexpr int kNoAllocMaxDevices = 64;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];
std::mutex g_noalloc_mutex;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// Unique id of the calling thread's current context (the runtime's primary context of
// the current device once a runtime call has made it current).
tcgStatus_t current_context_id(unsigned long long *id)
{
    if (!g_ctx_get_current || !g_ctx_get_id) {
        void *f1 = nullptr, *f2 = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault,
                                             &q1) != cudaSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault,
                                             &q2) != cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 ||
            !f2) {
            cudaGetLastError();
            return TCG_STATUS_NOT_INITIALIZED;
        }
        g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
        g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f2);
    }
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx || g_ctx_get_id(ctx, id) != CUDA_SUCCESS)
        return TCG_STATUS_NOT_INITIALIZED;
    return TCG_STATUS_SUCCESS;
}

// Once per device and context, with that device current: resolve the scratch and
// error-word addresses and the tensor-map encoder, and size the persistent grid.
tcgStatus_t noalloc_setup(int dev, NoAllocDevice **out)
{
    if (dev < 0 || dev >= kNoAllocMaxDevices)
        return TCG_STATUS_NOT_SUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    unsigned long long ctx_id = 0;
    tcgStatus_t cst = current_context_id(&ctx_id);
    if (cst != TCG_STATUS_SUCCESS) {
        // No context current on this thread yet: cudaSetDevice makes the device's
        // primary context current (it allocates nothing).
        if (cudaSetDevice(dev) != cudaSuccess) {
            cudaGetLastError();
            return TCG_STATUS_NOT_INITIALIZED;
        }
        cst = current_context_id(&ctx_id);
        if (cst != TCG_STATUS_SUCCESS)
            return cst;
    }
    NoAllocDevice &d = g_noalloc_dev[dev];
    if (!d.ready || d.ctx_id != ctx_id) {
        d.ready = false;
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return TCG_STATUS_NOT_INITIALIZED;
        }
        if (major != 10 || minor != 3)
            return TCG_STATUS_ARCH_MISMATCH;
        void *scratch = nullptr, *err = nullptr;
        if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess ||
            cudaGetSymbolAddress(&err, g_noalloc_err) != cudaSuccess || !scratch || !err) {
            cudaGetLastError();
            return TCG_STATUS_NOT_INITIALIZED;
        }
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
            cudaGetLastError();
            return TCG_STATUS_NOT_INITIALIZED;
        }
        d.scratch = scratch;
        d.err = static_cast<uint32_t *>(err);
        d.encode = reinterpret_cast<EncodeTiledFn>(fn);
        d.num_sms = sms;
        d.max_ctas = gemm_max_resident_ctas(2, sms);
        d.ctx_id = ctx_id;
        d.ready = true;
    }
    *out = &d;
    return TCG_STATUS_SUCCESS;
}

}  // namespace

extern "C" tcgStatus_t tcg_gemm_tf32_noalloc(void *stream, tcgOp_t transa, tcgOp_t transb,
                                             int64_t m, int64_t n, int64_t k, float alpha,
                                             const float *A, int64_t lda, const float *B,
                                             int64_t ldb, float beta, float *C, int64_t ldc)
{
    Problem p{transa, transb, m, n, k, alpha, beta, A, TCG_R_32F, lda, 0, B, TCG_R_32F, ldb, 0,
              C, TCG_R_32F, ldc, 0, 1, TCG_COMPUTE_32F_FAST_TF32, false};
    tcgStatus_t st = check_args(p);
    if (st != TCG_STATUS_SUCCESS || m == 0 || n == 0)
        return st;
    const bool product = k > 0 && alpha != 0.0f;
    if (product && tf32_ws_bytes(m, n, k, 1) > kNoAllocScratchBytes)
        return TCG_STATUS_NOT_SUPPORTED;     // operands do not fit the fixed scratch
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return TCG_STATUS_NOT_INITIALIZED;
    }
    NoAllocDevice *d = nullptr;
    st = noalloc_setup(dev, &d);
    if (st == TCG_STATUS_SUCCESS)
        st = device_ptr_ok(dev, C);
    if (st == TCG_STATUS_SUCCESS && product) {
        st = device_ptr_ok(dev, A);
        if (st == TCG_STATUS_SUCCESS)
            st = device_ptr_ok(dev, B);
    }
    if (st != TCG_STATUS_SUCCESS)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!product) {
        // D = beta*C: no operands, no scratch.
        int64_t blocks = (m * n + 255) / 256;
        const int64_t cap = static_cast<int64_t>(d->num_sms) * 8;
        if (blocks > cap)
            blocks = cap;
        return launch_scale(C, C, static_cast<int>(m), static_cast<int>(n), ldc, 0, 1, beta,
                            kOutF32, static_cast<int>(blocks), s) == cudaSuccess
                   ? TCG_STATUS_SUCCESS
                   : TCG_STATUS_EXECUTION_FAILED;
    }

    // A handle-like context on the stack: map encoding only, nothing allocated.
    tcgContext ctx;
    ctx.device = dev;
    ctx.num_sms = d->num_sms;
    ctx.encode = d->encode;

    // Round to TF32 into K-major copies inside the fixed scratch.
    const int kp = static_cast<int>((k + 3) / 4 * 4);
    uint8_t *Ak = static_cast<uint8_t *>(d->scratch);
    uint8_t *Bk = Ak + ((size_t)(m * kp) * 4 + 255) / 256 * 256;
    const bool a_kmajor = transa == TCG_OP_T, b_kmajor = transb == TCG_OP_N;
    const int grid_pack = d->num_sms * 8;
    if (launch_tf32_pack(A, lda, 0, a_kmajor ? 1 : 0, static_cast<int>(m), static_cast<int>(k), 1,
                         Ak, kp, m * kp, grid_pack, s) != cudaSuccess ||
        launch_tf32_pack(B, ldb, 0, b_kmajor ? 1 : 0, static_cast<int>(n), static_cast<int>(k), 1,
                         Bk, kp, n * kp, grid_pack, s) != cudaSuccess) {
        cudaGetLastError();
        return TCG_STATUS_EXECUTION_FAILED;
    }

    constexpr int cg = 2;
    GemmArgs a;
    std::memset(&a, 0, sizeof a);
    a.m = static_cast<int>(m); a.n = static_cast<int>(n); a.k = static_cast<int>(k); a.batch = 1;
    a.num_m_tiles = static_cast<int>((m + kBM * cg - 1) / (kBM * cg));
    a.num_n_tiles = static_cast<int>((n + kBN - 1) / kBN);
    a.k_row = 32;
    a.num_k_blocks = static_cast<int>((k + kDepth * 32 - 1) / (kDepth * 32));
    a.k_splits = 1;                              // never split: no partial-sum workspace
    a.kb_per_split = a.num_k_blocks;
    a.total_tiles = a.num_m_tiles * a.num_n_tiles;
    a.full_units = a.total_tiles;
    a.tail_splits = 1;
    a.tail_kb_per_split = a.num_k_blocks;
    a.group_m = 8;
    a.kind = kKindTF32;
    a.idesc = (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(kBN >> 3) << 17) |
              (static_cast<uint32_t>((kBM * cg) >> 4) << 24);
    a.alpha = alpha;
    a.beta = beta;
    a.c_bufs = beta == 0.0f ? 0 : (k * 4 <= 1024 * 4 ? 4 : 2);
    a.C = C;
    a.D = C;
    a.ldc = ldc;
    a.strideC = 0;
    a.err = d->err;
    a.wait_limit_ns = kDefaultWaitNs;
    CUtensorMap tmA, tmB;
    bool bca = false, bcb = false;
    st = operand_map(&ctx, Ak, TCG_R_32F, true, m, k, kp, m * kp, 1, kBM, a.k_row, &bca,
                     &a.a_mode, &tmA);
    if (st == TCG_STATUS_SUCCESS)
        st = operand_map(&ctx, Bk, TCG_R_32F, true, n, k, kp, n * kp, 1, kBN / cg, a.k_row, &bcb,
                         &a.b_mode, &tmB);
    if (st != TCG_STATUS_SUCCESS)
        return st;
    CUtensorMap tmD;
    st = output_map(&ctx, C, TCG_R_32F, m, n, ldc, 0, 1, &tmD, a.c_bufs);
    if (st != TCG_STATUS_SUCCESS)
        return st;
    const int64_t want = static_cast<int64_t>(a.total_tiles) * cg;
    const int grid = static_cast<int>(want < d->max_ctas ? want : d->max_ctas);
    if (launch_gemm(tmA, tmB, tmD, tmD, a, kOutF32, cg, kBN, grid, s) != cudaSuccess) {
        cudaGetLastError();
        return TCG_STATUS_EXECUTION_FAILED;
    }
    return TCG_STATUS_SUCCESS;
}

// The error word of the allocation-free calls: every bounded device wait that gave up
// since the last query has set a bit in it (it starts at zero when the library's module
// is loaded into a context).  Synchronises `stream` first so that the calls queued on it
// have finished, then reads and clears the word with plain symbol copies (nothing is
// allocated).
extern "C" tcgStatus_t tcg_noalloc_device_error(void *stream)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return TCG_STATUS_NOT_INITIALIZED;
    }
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return TCG_STATUS_EXECUTION_FAILED;
    }
    uint32_t bits = 0;
    if (cudaMemcpyFromSymbol(&bits, g_noalloc_err, sizeof bits) != cudaSuccess) {
        cudaGetLastError();
        return TCG_STATUS_EXECUTION_FAILED;
    }
    if (bits == 0)
        return TCG_STATUS_SUCCESS;
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_noalloc_err, &zero, sizeof zero) != cudaSuccess) {
        cudaGetLastError();
        return TCG_STATUS_EXECUTION_FAILED;
    }
    return TCG_STATUS_TIMEOUT;
}
