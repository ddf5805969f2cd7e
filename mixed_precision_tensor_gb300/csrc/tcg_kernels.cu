// tcg_kernels.cu -- device code of libtcg (sm_103a).
//
// tcg_gemm_kernel: persistent, warp-specialised tensor-core GEMM
//     D = alpha * op(A) * op(B) + beta * C
// ("Programming Tensor Cores in CUDA 9", sections "什么是张量核?" and "CUDA 9.0 中
// 张量核的编程访问": exact products, FP32 accumulation, alpha/beta applied to the
// accumulator elementwise; "CUDA Handbook, 17.5 Tensor Cores": one MMA instruction
// is a rank-K slab of the outer-product sum over k).
//
//   warp 0 (one lane)   TMA producer: per stage, one 128-byte row of K for every row of
//                        the CTA's A (128 rows) and B (128 rows per CTA of a pair, 256
//                        for a single CTA) into a ring of 128-byte-swizzled shared
//                        memory (6 stages of 32 KiB for a pair); out-of-range
//                        rows/columns/K are zero-filled by TMA, which makes ragged m, n,
//                        k exact.
//   warp 1 (one lane)   MMA issuer: tcgen05.mma (M=128 or 256 for a pair, N=256; K=16
//                        FP16/BF16, 8 TF32, 32 FP8) into a TMEM accumulator; two accumulators
//                        (2 x 256 columns) so the epilogue of tile t overlaps the
//                        main loop of tile t+1.  The page's diagnosis -- a tensor-core
//                        kernel that stalls waiting for the next slab ("CUDA Handbook,
//                        17.5", after Listing 17-5) -- is what the ring and the
//                        separate producer remove.
//   warps 2-9           epilogue: tcgen05.ld TMEM -> registers, alpha*acc + beta*C in
//                        FP32 (C by TMA), round to the output type (nearest even) into a
//                        staging buffer, TMA store of D.
//
// Every wait is bounded (globaltimer): a wait that runs out sets a bit in the device
// error word and a shared abort flag, every role stops, in-flight copies and MMAs are
// drained, TMEM is freed and the kernel returns.  No trap, no unbounded spin.
//
// tcg_scale_kernel: D = beta * C (k == 0 or alpha == 0, A and B not read).
// tcg_splitk_reduce_kernel / tcg_tail_reduce_kernel: K-range partial sums added in
// range order, then alpha, beta and the output rounding.
// tcg_tf32_round_kernel / tcg_tf32_transpose_round_kernel / tcg_tf32_pack_kernel:
// FP32 -> TF32 (round to nearest even) into K-major copies.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "tcg_internal.h"
#include "tcg_ptx.cuh"

namespace tcg {

constexpr int kMaxStages = TileCfg<2, 0, kBNNarrow>::kStages;
constexpr int kMaxEpiBufs = 4;

struct SmemCtl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t acc_full[kMaxAccBufs];
    uint64_t acc_empty[kMaxAccBufs];
    uint64_t c_full[2][kMaxEpiBufs];   // epilogue half x staging buffer: C chunk landed
    uint64_t drain;
    uint32_t tmem_base;
    volatile int abort_flag;
    volatile int cv_slot[2];           // epilogue half: the sub-unit its leader claimed
};
static_assert(sizeof(SmemCtl) <= kBarrierBytes, "barrier area too small");

// Raise the abort flag in this CTA and, for a pair, in the peer CTA.
template <int CG>
__device__ __forceinline__ void raise_abort(SmemCtl *ctl, const GemmArgs &p, uint32_t err_bit)
{
    ctl->abort_flag = 1;
    if constexpr (CG == 2)
        st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int *>(&ctl->abort_flag)),
                                          cluster_ctarank() ^ 1u),
                              1u);
    atomicOr(p.err, err_bit);
}

// Bounded wait on an mbarrier phase.  Returns false if the kernel was aborted or the
// limit ran out (then the error bit is recorded and the abort flag raised).
template <int CG>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, SmemCtl *ctl,
                                             const GemmArgs &p, uint32_t err_bit,
                                             bool honour_abort = true)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (honour_abort && ctl->abort_flag)
            return false;
        if (globaltimer_ns() - t0 > p.wait_limit_ns) {
            raise_abort<CG>(ctl, p, err_bit);
            return false;
        }
    }
}


// Work unit u -> its tile (b, mt, nt), its K blocks [kb0, kb1), and -- for a unit of a
// split tail tile -- its partial-sum slice (-1 otherwise).  Units [0, full_units) are
// tiles u / k_splits with K range u % k_splits (k_splits = 1: whole tiles); the units
// after them are the tail tiles full_units, full_units + 1, ..., tail_splits units each.
struct UnitInfo {
    int b, mt, nt, kb0, kb1, ks, tail_slice;
};
__device__ __forceinline__ UnitInfo unit_info(const GemmArgs &p, int u)
{
    UnitInfo w;
    int t, s, kbps;
    if (u < p.full_units) {
        t = u / p.k_splits;
        s = u - t * p.k_splits;
        kbps = p.kb_per_split;
        w.tail_slice = -1;
    } else {
        const int v = u - p.full_units;
        const int r = v / p.tail_splits;
        s = v - r * p.tail_splits;
        t = p.full_units + r;
        kbps = p.tail_kb_per_split;
        w.tail_slice = v;
    }
    raster(p, t, w.b, w.mt, w.nt);
    w.ks = s;
    w.kb0 = s * kbps;
    w.kb1 = min(w.kb0 + kbps, p.num_k_blocks);
    return w;
}

// FP32 -> TF32, round to nearest, ties to even, kept in FP32 bits (low 13 bits zero).
// Inf passes through; NaN becomes a quiet NaN of the same sign (its payload could sit
// entirely in the 13 dropped bits).  A carry out of the mantissa moves to the next
// binade, and values past the largest TF32 number become Inf, as RNE requires.
__device__ __forceinline__ uint32_t tf32_rne_bits(uint32_t u)
{
    if ((u & 0x7F800000u) == 0x7F800000u)
        return (u & 0x007FFFFFu) ? ((u & 0x80000000u) | 0x7FC00000u) : u;
    return (u + 0x0FFFu + ((u >> 13) & 1u)) & 0xFFFFE000u;
}

// Two-word TF32 split of an FP32 value ("NVIDIA Tensor Core混合精度计算原理与应用解析",
// section 5.1: represent each operand by pieces the tensor core multiplies exactly):
// hi = RNE_tf32(x), lo = RNE_tf32(x - hi).  x - hi is exact in FP32 (hi is within a
// factor of two of x), so x = hi + lo up to 2^-22 |x|.  Inf and NaN keep hi = x, lo = 0;
// a finite x that rounds past the largest TF32 value is truncated instead, so hi stays
// finite and lo carries the rest.
__device__ __forceinline__ void tf32_split_bits(uint32_t u, uint32_t &hi, uint32_t &lo)
{
    hi = tf32_rne_bits(u);
    if ((u & 0x7F800000u) == 0x7F800000u) {
        lo = 0u;
        return;
    }
    if ((hi & 0x7F800000u) == 0x7F800000u)
        hi = u & 0xFFFFE000u;
    lo = tf32_rne_bits(__float_as_uint(__uint_as_float(u) - __uint_as_float(hi)));
}

// ------------------------------------------ TF32 rounding inside the GEMM kernel
// kKindTF32R: the GEMM kernel writes the rounded K-major copies of op(A) and op(B) itself
// while it multiplies, instead of two pre-pass kernels running before it.  The copies
// are cut into items (operand, batch entry, panel of tile rows, chunk of K) and the
// items into sub-units of kCvRows x kCvK elements (GemmArgs cv_*).  The epilogue warps,
// idle while an accumulator fills, claim sub-units through a per-item counter, in the
// order in which their own pair's work units will need them, round them and count them
// done; the producer waits for an item's count before it loads the item's stages.  Each
// element is rounded once, so the extra traffic is one read and one write of each
// operand, spread over the GEMM, where the pre-pass kernels ran alone before it.
// Nothing inside a sub-unit waits, so a claimed sub-unit always completes, and every
// item a pair needs lies on its own walk: the producers' waits end whether or not the
// other CTAs are resident.

struct CvItem {
    int x, b, panel, chunk;
};
__device__ __forceinline__ CvItem cv_item(const GemmArgs &p, int item)
{
    CvItem it;
    it.x = item >= p.cv_base[1] ? 1 : 0;
    const int rem = item - p.cv_base[it.x];
    const int bp = rem / p.cv_chunks;
    it.chunk = rem - bp * p.cv_chunks;
    it.b = bp / p.cv_panels[it.x];
    it.panel = bp - it.b * p.cv_panels[it.x];
    return it;
}

// Round sub-unit s of an item with the 128 threads of an epilogue half (tid = 0..127,
// named barrier bar_id); tile: 16 KiB of the half's staging buffer.  Sub-unit s covers
// rows r0 .. r0 + 63 of the panel and K elements q0 .. q0 + 127 of the chunk.
//   K-major source: 32 threads per row (16 bytes each), 16 rows per thread, read and
//     written along K.
//   M/N-major source: two 64 x 64 transposes through shared memory, 16 threads per
//     64-element row on both sides (16-byte global accesses).  The tile has no padding
//     column: element (K row kr, row r) sits at word kr * 64 + (r ^ 2 (kr >> 2)), which
//     keeps the 16-byte writes and the 4-byte column reads free of bank conflicts.
// As in the pre-pass kernels, rows past the operand are skipped, K past k reads zeros
// (M/N-major) and each 16-byte group that starts before round_up(k, 4) is written.
// mid() runs once every load is issued: the half's leader uses it to overlap its
// bookkeeping (the previous sub-unit's done count, the next claim) with the loads.
template <bool kSplit, typename Mid>
__device__ __forceinline__ void cv_convert(const GemmArgs &p, int item, int s, int tid,
                                           uint32_t *tile, uint32_t bar_id, Mid &&mid)
{
    const CvItem it = cv_item(p, item);
    const int x = it.x;
    const int rg = p.cv_panel_rows[x] / kCvRows;
    const int r0 = it.panel * p.cv_panel_rows[x] + (s % rg) * kCvRows;
    const int64_t q0 = static_cast<int64_t>(it.chunk) * p.cv_kc + (s / rg) * kCvK;
    const int rows = p.cv_rows[x];
    const int64_t kp = p.cv_kp, ld = p.cv_ld[x];
    const uint32_t *src = static_cast<const uint32_t *>(p.cv_src[x]) + it.b * p.cv_stride[x];
    uint32_t *dst = static_cast<uint32_t *>(p.cv_dst[x]) + it.b * p.cv_dstride[x];
    uint32_t *dst_lo = kSplit ? static_cast<uint32_t *>(p.cv_dst_lo[x]) + it.b * p.cv_dstride[x]
                              : nullptr;
    // RNE to TF32, or (two-word split) the high word with the low word written beside it
    auto put = [&](int64_t off, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
        if constexpr (kSplit) {
            uint4 hi, lo;
            tf32_split_bits(a, hi.x, lo.x);
            tf32_split_bits(b, hi.y, lo.y);
            tf32_split_bits(c, hi.z, lo.z);
            tf32_split_bits(d, hi.w, lo.w);
            *reinterpret_cast<uint4 *>(dst + off) = hi;
            *reinterpret_cast<uint4 *>(dst_lo + off) = lo;
        } else {
            *reinterpret_cast<uint4 *>(dst + off) =
                make_uint4(tf32_rne_bits(a), tf32_rne_bits(b), tf32_rne_bits(c), tf32_rne_bits(d));
        }
    };
    if (p.cv_kmajor[x]) {
        const int j = tid & 31, rr = tid >> 5;
        const int64_t q = q0 + 4 * j;
        uint4 v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int r = r0 + rr + 4 * i;
            v[i] = make_uint4(0u, 0u, 0u, 0u);
            if (r < rows && q < kp)
                v[i] = __ldg(reinterpret_cast<const uint4 *>(src + q + static_cast<int64_t>(r) * ld));
        }
        mid();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int r = r0 + rr + 4 * i;
            if (r < rows && q < kp)
                put(q + static_cast<int64_t>(r) * kp, v[i].x, v[i].y, v[i].z, v[i].w);
        }
        return;
    }
    const int k = p.k;
    const int c = tid & 15, w = tid >> 4;
    uint4 v[2][8];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int j = 0; j < 8; ++j) {           // K rows q0 + 64 t + w + 8 j, rows r0 + 4c ..
            const int64_t q = q0 + 64 * t + w + 8 * j;
            const int r = r0 + 4 * c;
            v[t][j] = make_uint4(0u, 0u, 0u, 0u);
            if (q < k && r < rows)
                v[t][j] = __ldg(reinterpret_cast<const uint4 *>(src + r + q * ld));
        }
    mid();
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        named_barrier_sync(bar_id, 128);         // the tile's previous readers are done
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int kr = w + 8 * j;
            const uint32_t f = static_cast<uint32_t>(kr >> 2) << 1;
            // words 4c .. 4c + 3 of K row kr go to 4 (c ^ (f >> 2)) + (i ^ (f & 2))
            const uint4 u = v[t][j];
            const uint4 o = (f & 2u) ? make_uint4(u.z, u.w, u.x, u.y) : u;
            *reinterpret_cast<uint4 *>(tile + kr * 64 + 4 * (c ^ static_cast<int>(f >> 2))) = o;
        }
        named_barrier_sync(bar_id, 128);
        const int64_t q = q0 + 64 * t + 4 * c;
#pragma unroll
        for (int j = 0; j < 8; ++j) {             // output rows r0 + w + 8 j
            const int rl = w + 8 * j, r = r0 + rl;
            if (r >= rows || q >= k)
                continue;
            const int sw = rl ^ (2 * c);
            put(q + static_cast<int64_t>(r) * kp, tile[(4 * c) * 64 + sw],
                tile[(4 * c + 1) * 64 + sw], tile[(4 * c + 2) * 64 + sw],
                tile[(4 * c + 3) * 64 + sw]);
        }
    }
}

// The producer's wait for items ia and ib (their sub-units done), bounded like every
// wait of the kernel; then this thread's TMA loads see the rounded values.
template <int CG>
__device__ __forceinline__ bool cv_wait(const GemmArgs &p, SmemCtl *ctl, int ia, int ib)
{
    const uint32_t *done = p.cv_cnt + p.cv_items;
    const uint32_t ta = static_cast<uint32_t>(p.cv_subs[0]);
    const uint32_t tb = static_cast<uint32_t>(p.cv_subs[1]);
    if (ld_relaxed_gpu(done + ia) < ta || ld_relaxed_gpu(done + ib) < tb) {
        const uint64_t t0 = globaltimer_ns();
        while (ld_relaxed_gpu(done + ia) < ta || ld_relaxed_gpu(done + ib) < tb) {
            if (ctl->abort_flag)
                return false;
            if (globaltimer_ns() - t0 > p.wait_limit_ns) {
                raise_abort<CG>(ctl, p, kErrConvert);
                return false;
            }
        }
    }
    fence_acq_rel_gpu();
    fence_proxy_async_global();
    return true;
}

// Count sub-units of `item` done (the half's leader, after a barrier that follows every
// thread's writes of it): the fence makes those writes visible at GPU scope before the
// counts (the barrier-then-fence release pattern).
__device__ __forceinline__ void cv_report(const GemmArgs &p, int item)
{
    const CvItem ci = cv_item(p, item);
    __threadfence();
    atomicAdd(p.cv_cnt + p.cv_items + item, 1u);
    atomicAdd(p.cv_cnt + 2 * p.cv_items + p.cv_pbase[ci.x] + ci.b * p.cv_panels[ci.x] + ci.panel,
              1u);
}

// An epilogue half's walk over the items its pair's work units need, in the order they
// need them: unit by unit (t = cluster_id, + num_clusters, ...), chunk by chunk, A then
// B.  claim() returns item * 64 + sub-unit of the next sub-unit it won, or -1 once the
// walk is over.  Only the half's leader walks.
struct CvWalk {
    int t, c, c_end, x, ia, ib;

    __device__ __forceinline__ void start(const GemmArgs &p, int unit)
    {
        t = unit;
        x = 0;
        if (t >= p.total_tiles)
            return;
        const UnitInfo w = unit_info(p, t);
        const int kstage = kDepth * (kRowBytes / 4);            // K elements per stage
        c = (w.kb0 * kstage) / p.cv_kc;
        c_end = (w.kb1 * kstage + p.cv_kc - 1) / p.cv_kc;
        ia = p.cv_base[0] + ((p.a_bcast ? 0 : w.b) * p.cv_panels[0] + w.mt) * p.cv_chunks;
        ib = p.cv_base[1] + ((p.b_bcast ? 0 : w.b) * p.cv_panels[1] + w.nt) * p.cv_chunks;
    }

    __device__ __forceinline__ int claim(const GemmArgs &p, int num_clusters)
    {
        uint32_t *claimed = p.cv_cnt;
        while (t < p.total_tiles) {
            const int item = (x == 0 ? ia : ib) + c;
            const uint32_t subs = static_cast<uint32_t>(p.cv_subs[x]);
            if (ld_relaxed_gpu(claimed + item) < subs) {
                const uint32_t s = atomicAdd(claimed + item, 1u);
                if (s < subs)
                    return item * 64 + static_cast<int>(s);
            }
            if (x == 0) {
                x = 1;
            } else if (++c < c_end) {
                x = 0;
            } else {
                start(p, t + num_clusters);
            }
        }
        return -1;
    }
};

template <int OUT>
__device__ __forceinline__ void store_out(void *D, int64_t idx, float v)
{
    if constexpr (OUT == kOutF32)
        static_cast<float *>(D)[idx] = v;
    else if constexpr (OUT == kOutF16)
        static_cast<__half *>(D)[idx] = __float2half_rn(v);
    else
        static_cast<__nv_bfloat16 *>(D)[idx] = __float2bfloat16_rn(v);
}

template <int OUT>
__device__ __forceinline__ float load_smem(const uint8_t *buf, int idx)
{
    if constexpr (OUT == kOutF32)
        return reinterpret_cast<const float *>(buf)[idx];
    else if constexpr (OUT == kOutF16)
        return __half2float(reinterpret_cast<const __half *>(buf)[idx]);
    else
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(buf)[idx]);
}

template <int OUT>
__device__ __forceinline__ void store_smem(uint8_t *buf, int idx, float v)
{
    if constexpr (OUT == kOutF32)
        reinterpret_cast<float *>(buf)[idx] = v;
    else if constexpr (OUT == kOutF16)
        reinterpret_cast<__half *>(buf)[idx] = __float2half_rn(v);
    else
        reinterpret_cast<__nv_bfloat16 *>(buf)[idx] = __float2bfloat16_rn(v);
}

// Two elements of one row, columns idx and idx + stride of the staging buffer, rounded to
// the 16-bit output type (nearest even) by one packed conversion (cvt.rn.f16x2.f32 /
// cvt.rn.bf16x2.f32): the same values as two scalar conversions, in half the
// instructions.
template <int OUT>
__device__ __forceinline__ void store_smem_pair(uint8_t *buf, int idx, int stride, float a, float b)
{
    uint32_t packed;
    if constexpr (OUT == kOutF16) {
        const __half2 h = __floats2half2_rn(a, b);
        packed = *reinterpret_cast<const uint32_t *>(&h);
    } else {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        packed = *reinterpret_cast<const uint32_t *>(&h);
    }
    uint16_t *q = reinterpret_cast<uint16_t *>(buf);
    q[idx] = static_cast<uint16_t>(packed & 0xFFFFu);
    q[idx + stride] = static_cast<uint16_t>(packed >> 16);
}

template <int OUT>
__device__ __forceinline__ float load_c(const void *C, int64_t idx)
{
    if constexpr (OUT == kOutF32)
        return static_cast<const float *>(C)[idx];
    else if constexpr (OUT == kOutF16)
        return __half2float(static_cast<const __half *>(C)[idx]);
    else
        return __bfloat162float(static_cast<const __nv_bfloat16 *>(C)[idx]);
}

// CG = 1: one CTA per 128x256 tile.  CG = 2: a CTA pair (cluster of 2) per 256x256 tile;
// the even CTA issues the MMAs (cta_group::2), both CTAs load their halves of A and B
// and signal the even CTA's "full" barrier, the MMA completion is multicast to both
// CTAs' "empty" and "accumulator full" barriers, and both CTAs' epilogues report to the
// even CTA's "accumulator empty" barrier.
template <int OUT, int CG, int KIND, int CBUF, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    tcg_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmD,
                    const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ CUtensorMap tmA2,
                    const __grid_constant__ CUtensorMap tmB2, const GemmArgs p)
{
    constexpr int kOutB = OUT == kOutF32 ? 4 : 2;
    constexpr int kChunkB = epi_chunk_bytes(kOutB, CBUF);   // bytes of one epilogue chunk
    using Cfg = TileCfg<CG, CBUF, BN, kChunkB>;
    constexpr int kAccBufs = Cfg::kAccBufs;
    constexpr bool BETA = CBUF != 0;                          // C is read
    // Two-word TF32 (kKindTF32x3): a stage carries A's and B's high words, then their
    // low words (tmA2, tmB2); each K slice takes three products, lo_A hi_B, hi_A lo_B and
    // hi_A hi_B, into the one accumulator.
    constexpr bool kX3 = KIND == kKindTF32x3 || KIND == kKindTF32x3R;
    // In-kernel TF32 rounding (kKindTF32R): the epilogue warps round the operands into
    // their K-major copies between accumulators and the producer waits for each item.
    constexpr bool kFuse = KIND == kKindTF32R || KIND == kKindTF32x3R;
    constexpr int kOps = kX3 ? 2 : 1;                         // words per operand
    constexpr int kStages = Cfg::kRingBytes / (kOps * Cfg::kStageBytes);
    static_assert(kStages >= 2, "ring too small");
    constexpr int kRingBytes = Cfg::kRingBytes;
    constexpr int kEpiBufs = Cfg::kEpiBufs;
    constexpr int kEpiBytes = Cfg::kEpiBytes;
    constexpr int kBRows = Cfg::kBRows;
    constexpr int kAStage = Cfg::kAStage;
    constexpr int kBStage = Cfg::kBStage;
    constexpr int kStageBytes = kOps * Cfg::kStageBytes;     // all words of A and B
    constexpr int kTileM = Cfg::kTileM;

    unsigned long long clk0 = 0, ns0 = 0;
    if (p.clk && threadIdx.x == 0) {
        clk0 = clock64();
        ns0 = globaltimer_ns();
    }
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms.
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw_u32);
    const uint32_t a_smem = base;
    const uint32_t b_smem = base + kStages * kAStage;
    const uint32_t a2_smem = b_smem + kStages * kBStage;    // low words (kX3)
    const uint32_t b2_smem = a2_smem + kStages * kAStage;
    const uint32_t epi_smem = base + kRingBytes;
    uint8_t *epi_ptr = base_ptr + kRingBytes;
    SmemCtl *ctl = reinterpret_cast<SmemCtl *>(base_ptr + kRingBytes + kEpiBytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = (CG == 2) ? cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int cluster_id = blockIdx.x / CG;
    const int num_clusters = gridDim.x / CG;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int a = 0; a < kAccBufs; ++a) {
            mbar_init(smem_u32(&ctl->acc_full[a]), 1);
            mbar_init(smem_u32(&ctl->acc_empty[a]), kEpiWarps * CG);
        }
        for (int h = 0; h < 2; ++h)
            for (int bf = 0; bf < kEpiBufs; ++bf)
                mbar_init(smem_u32(&ctl->c_full[h][bf]), 1);
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        tma_prefetch_map(&tmD);
        if constexpr (kX3) {
            tma_prefetch_map(&tmA2);
            tma_prefetch_map(&tmB2);
        }
        if (p.tail_splits > 1)
            tma_prefetch_map(&tmW);
    }
    __syncwarp();
    if (warp == 1) {
        if constexpr (CG == 2) {
            tmem_alloc_pair(smem_u32(&ctl->tmem_base), kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    if constexpr (CG == 2)
        cluster_sync_all();
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    // Chained calls: the set-up above (barriers, TMEM, tensor-map prefetch) may overlap the
    // end of the previous kernel on the stream; nothing below touches global memory before
    // that kernel has completed and its writes are visible.
    if (threadIdx.x == 0)
        griddep_launch_dependents();
    griddep_wait();

    // The MMA kind is a template argument and every per-slice descriptor offset is
    // computed before the loop: the issuing thread's loop must stay branch-free and
    // short, as its instruction rate is what keeps the tensor core fed.
    constexpr bool kTf32 = KIND == kKindTF32 || kX3 || kFuse;
    constexpr uint32_t kEsize = kTf32 ? 4u : (KIND == kKindF8 ? 1u : 2u);
    constexpr uint32_t kKmma = 32u / kEsize;                  // K per MMA instruction
    constexpr int kMmasPerRow = kRowBytes / 32;               // 4 MMAs per 128-byte K row
    constexpr int kMmasPerStage = kMmasPerRow * kDepth;       // 4
    constexpr int kKRow = kRowBytes / kEsize;                 // K elements per 128-byte row
    constexpr int kMnBox = kRowBytes / kEsize;                // M/N elements per 128-byte chunk
    // Bytes of one kMnBox-element chunk of an M/N-major operand: kDepth K rows each.
    constexpr uint32_t kChunkBytes = kDepth * kKRow * kRowBytes;
    // Per operand (see OperandMode): the descriptor's leading / stride byte offsets and
    // the byte offset of K slice j (one MMA) inside a stage.
    //   kK:  slice j = K row j / 4 (a box of rows x 128 B), 32 bytes per slice within it;
    //        8-row groups 1 KiB apart (SBO); LBO unused.
    //   kMN: kKmma K rows of 128 B per slice, all chunks at once: LBO = chunk stride,
    //        SBO = next 8-row K group (1 KiB).
    auto layout = [&](int mode, int rows, uint32_t &lbo, uint32_t &sbo, uint32_t *off) {
        sbo = 8 * kRowBytes;
        lbo = mode == kK ? 16u : kChunkBytes;
#pragma unroll
        for (int j = 0; j < kMmasPerStage; ++j) {
            const uint32_t b = mode == kK
                ? static_cast<uint32_t>((j / kMmasPerRow) * rows * kRowBytes + (j % kMmasPerRow) * 32)
                : static_cast<uint32_t>(j) * kKmma * kRowBytes;
            off[j] = b >> 4;                                   // descriptor address units
        }
    };
    uint32_t a_lbo, a_sbo, b_lbo, b_sbo, a_off[kMmasPerStage], b_off[kMmasPerStage];
    layout(p.a_mode, kBM, a_lbo, a_sbo, a_off);
    layout(p.b_mode, kBRows, b_lbo, b_sbo, b_off);
    // Descriptors of stage 0, K slice 0; other slices add (byte offset >> 4) to the
    // start-address field (bits 0-13), which cannot overflow in 227 KB of shared memory.
    const uint64_t a_desc0 = smem_desc_sw128(a_smem, a_lbo, a_sbo);
    const uint64_t b_desc0 = smem_desc_sw128(b_smem, b_lbo, b_sbo);
    const uint64_t a2_desc0 = smem_desc_sw128(a2_smem, a_lbo, a_sbo);
    const uint64_t b2_desc0 = smem_desc_sw128(b2_smem, b_lbo, b_sbo);
    uint32_t issued_mask = 0, issued_parity = 0;              // leader producer: loads per stage

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ producer
            int stage = 0;
            uint32_t phase = 0;
            bool skip_once = p.fault_inject != 0 && leader;
            bool ok = true;
            // Operands that exactly one tile reads (p.a_once / p.b_once) are loaded with
            // L2 evict_first, so that they do not displace data that is read again.
            const uint64_t pol_a = l2_policy(p.a_once != 0);
            const uint64_t pol_b = l2_policy(p.b_once != 0);
            for (int t = cluster_id; ok && t < p.total_tiles; t += num_clusters) {
                const UnitInfo w = unit_info(p, t);
                const int kb_begin = w.kb0, kb_end = w.kb1;
                const int m0 = w.mt * kTileM + static_cast<int>(rank) * kBM;
                const int n0 = w.nt * BN + static_cast<int>(rank) * kBRows;
                const int za = p.a_bcast ? 0 : w.b, zb = p.b_bcast ? 0 : w.b;
                // In-kernel rounding: the unit's items (A and B, chunk 0 of the panel); when
                // both panels are done already, the unit needs no further waits.
                int cv_ia = 0, cv_ib = 0;
                bool cv_ready = true;
                if constexpr (kFuse) {
                    cv_ia = p.cv_base[0] + (za * p.cv_panels[0] + w.mt) * p.cv_chunks;
                    cv_ib = p.cv_base[1] + (zb * p.cv_panels[1] + w.nt) * p.cv_chunks;
                    const uint32_t *pdone = p.cv_cnt + 2 * p.cv_items;
                    const int pa = p.cv_pbase[0] + za * p.cv_panels[0] + w.mt;
                    const int pb = p.cv_pbase[1] + zb * p.cv_panels[1] + w.nt;
                    cv_ready = ld_relaxed_gpu(pdone + pa) >=
                                   static_cast<uint32_t>(p.cv_subs[0] * p.cv_chunks) &&
                               ld_relaxed_gpu(pdone + pb) >=
                                   static_cast<uint32_t>(p.cv_subs[1] * p.cv_chunks);
                    if (cv_ready) {
                        fence_acq_rel_gpu();
                        fence_proxy_async_global();
                    }
                }
                // The unit's K loop; `hinted` selects the loads with an L2 cache policy
                // (operands read once), outside the loop so that the common path keeps the
                // plain loads (the policy operand cost ~1.3% on tensor-bound problems).
                auto k_loop = [&](auto hinted) {
                    for (int kb = kb_begin; kb < kb_end; ++kb) {
                        if constexpr (kFuse) {
                            if (!cv_ready && (kb == kb_begin || kb % p.cv_kb_per_chunk == 0)) {
                                const int c = kb / p.cv_kb_per_chunk;
                                if (!cv_wait<CG>(p, ctl, cv_ia + c, cv_ib + c)) {
                                    ok = false;
                                    break;
                                }
                            }
                        }
                        const uint32_t fb_local = smem_u32(&ctl->full[stage]);
                        const uint32_t fb = (CG == 2) ? mapa_shared(fb_local, 0) : fb_local;
                        if (!wait_bounded<CG>(smem_u32(&ctl->empty[stage]), phase ^ 1u, ctl, p,
                                              kErrProducer)) {
                            ok = false;
                            break;
                        }
                        if (skip_once) {
                            skip_once = false;  // test hook: this stage is never filled
                        } else {
                            if (leader) {
                                mbar_arrive_expect_tx(fb_local, kStageBytes * CG);
                                issued_mask |= 1u << stage;
                                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                            }
                            const uint32_t sa = a_smem + stage * kAStage;
                            const uint32_t sb = b_smem + stage * kBStage;
                            const int k0 = kb * kDepth * kKRow;
                            // One operand tile: `rows` rows starting at row0, K from k0: kDepth
                            // boxes of rows x 128 B (K-major), one 4-D box holding every
                            // c-element chunk of rows (M/N-major, kMN4) or one box per chunk
                            // (M/N-major with ragged rows, kMN); chunks cover all kDepth K rows.
                            auto box = [&](uint32_t d, const CUtensorMap *map, int x, int y, int z,
                                           uint64_t pol) {
                                if constexpr (decltype(hinted)::value) {
                                    if constexpr (CG == 2)
                                        tma_load_3d_pair_hint(d, map, fb, x, y, z, pol);
                                    else
                                        tma_load_3d_hint(d, map, fb, x, y, z, pol);
                                } else {
                                    if constexpr (CG == 2)
                                        tma_load_3d_pair(d, map, fb, x, y, z);
                                    else
                                        tma_load_3d(d, map, fb, x, y, z);
                                }
                            };
                            auto load = [&](uint32_t dst, const CUtensorMap *map, int mode, auto rows_c,
                                            int row0, int z, uint64_t pol) {
                                constexpr int kRows = decltype(rows_c)::value;
                                if (mode == kK) {
#pragma unroll
                                    for (int h = 0; h < kDepth; ++h)
                                        box(dst + h * kRows * kRowBytes, map, k0 + h * kKRow, row0, z,
                                            pol);
                                } else if (mode == kMN4) {
                                    if constexpr (decltype(hinted)::value) {
                                        if constexpr (CG == 2)
                                            tma_load_4d_pair_hint(dst, map, fb, 0, k0, row0 / kMnBox,
                                                                  z, pol);
                                        else
                                            tma_load_4d_hint(dst, map, fb, 0, k0, row0 / kMnBox, z,
                                                             pol);
                                    } else {
                                        if constexpr (CG == 2)
                                            tma_load_4d_pair(dst, map, fb, 0, k0, row0 / kMnBox, z);
                                        else
                                            tma_load_4d(dst, map, fb, 0, k0, row0 / kMnBox, z);
                                    }
                                } else {
#pragma unroll
                                    for (int h = 0; h < kRows / kMnBox; ++h)
                                        box(dst + h * kChunkBytes, map, row0 + h * kMnBox, k0, z, pol);
                                }
                            };
                            load(sa, &tmA, p.a_mode, std::integral_constant<int, kBM>{}, m0, za, pol_a);
                            load(sb, &tmB, p.b_mode, std::integral_constant<int, kBRows>{}, n0, zb,
                                 pol_b);
                            if constexpr (kX3) {
                                load(a2_smem + stage * kAStage, &tmA2, p.a_mode,
                                     std::integral_constant<int, kBM>{}, m0, za, pol_a);
                                load(b2_smem + stage * kBStage, &tmB2, p.b_mode,
                                     std::integral_constant<int, kBRows>{}, n0, zb, pol_b);
                            }
                        }
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                };
                if (p.a_once || p.b_once)
                    k_loop(std::true_type{});
                else
                    k_loop(std::false_type{});
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ----------------------------------------------------------- MMA issue
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int t = cluster_id; ok && t < p.total_tiles; t += num_clusters, ++it) {
                const UnitInfo w = unit_info(p, t);
                const int kb_begin = w.kb0, kb_end = w.kb1;
                const int acc = it % kAccBufs;
                const uint32_t acc_phase = (it / kAccBufs) & 1;
                if (!wait_bounded<CG>(smem_u32(&ctl->acc_empty[acc]), acc_phase ^ 1u, ctl, p,
                                      kErrMmaAcc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    if (!wait_bounded<CG>(smem_u32(&ctl->full[stage]), phase, ctl, p,
                                          kErrMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad_s = a_desc0 + ((static_cast<uint32_t>(stage) * kAStage) >> 4);
                    const uint64_t bd_s = b_desc0 + ((static_cast<uint32_t>(stage) * kBStage) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kMmasPerStage; ++kk) {
                        const uint64_t ad = ad_s + a_off[kk];
                        const uint64_t bd = bd_s + b_off[kk];
                        const uint32_t accum = (kb > kb_begin || kk > 0) ? 1u : 0u;
                        if constexpr (kX3) {
                            // the two small products first, then hi_A hi_B
                            const uint64_t ad2 = a2_desc0 +
                                ((static_cast<uint32_t>(stage) * kAStage) >> 4) + a_off[kk];
                            const uint64_t bd2 = b2_desc0 +
                                ((static_cast<uint32_t>(stage) * kBStage) >> 4) + b_off[kk];
                            if constexpr (CG == 2) {
                                mma_tf32_pair(d_tmem, ad2, bd, p.idesc, accum);
                                mma_tf32_pair(d_tmem, ad, bd2, p.idesc, 1u);
                                mma_tf32_pair(d_tmem, ad, bd, p.idesc, 1u);
                            } else {
                                mma_tf32(d_tmem, ad2, bd, p.idesc, accum);
                                mma_tf32(d_tmem, ad, bd2, p.idesc, 1u);
                                mma_tf32(d_tmem, ad, bd, p.idesc, 1u);
                            }
                        } else if constexpr (CG == 2) {
                            if constexpr (KIND == kKindTF32 || kFuse)
                                mma_tf32_pair(d_tmem, ad, bd, p.idesc, accum);
                            else if constexpr (KIND == kKindF8)
                                mma_f8_pair(d_tmem, ad, bd, p.idesc, accum);
                            else
                                mma_f16_pair(d_tmem, ad, bd, p.idesc, accum);
                        } else {
                            if constexpr (KIND == kKindTF32 || kFuse)
                                mma_tf32(d_tmem, ad, bd, p.idesc, accum);
                            else if constexpr (KIND == kKindF8)
                                mma_f8(d_tmem, ad, bd, p.idesc, accum);
                            else
                                mma_f16(d_tmem, ad, bd, p.idesc, accum);
                        }
                    }
                    // the stage is free (in both CTAs) once these MMAs have read it
                    if constexpr (CG == 2)
                        mma_commit_pair_mc(smem_u32(&ctl->empty[stage]), 0x3);
                    else
                        mma_commit(smem_u32(&ctl->empty[stage]));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                // accumulator ready (in both CTAs)
                if constexpr (CG == 2)
                    mma_commit_pair_mc(smem_u32(&ctl->acc_full[acc]), 0x3);
                else
                    mma_commit(smem_u32(&ctl->acc_full[acc]));
            }
            // Every MMA issued so far must be complete before TMEM is released.
            if constexpr (CG == 2)
                mma_commit_pair(smem_u32(&ctl->drain));
            else
                mma_commit(smem_u32(&ctl->drain));
            wait_bounded<CG>(smem_u32(&ctl->drain), 0, ctl, p, kErrDrain, false);
        }
    } else {
        // -------------------------------------------------------------- epilogue
        // Two halves of 4 warps; half h owns TMEM columns [h BN/2, (h + 1) BN/2) of each tile
        // for all 128 rows (warp w reads TMEM lane quarter w % 4), in chunks of kCols
        // columns.  Per chunk: C (with beta != 0) lands by TMA in a staging buffer, every
        // thread combines its row with the accumulator in place (the buffer is a
        // column-major 128 x kCols block of D), and the half's leader writes the block to
        // D with one TMA store, which clips rows >= m and columns >= n.  The chunks of all
        // tiles form one sequence g = 0, 1, ... per half; with beta != 0 the C loads run
        // kEpiBufs - 1 chunks ahead of it (across tile boundaries).
        constexpr int kOutBytes = OUT == kOutF32 ? 4 : 2;
        constexpr int kCols = epi_cols(kOutBytes, CBUF);       // 16 (FP32), 32 or 64 (16-bit)
        constexpr int kChunks = (BN / 2) / kCols;              // per half per tile
        constexpr int kAhead = BETA ? kEpiBufs - 1 : 0;        // C loads in flight
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        const bool half_leader = (warp == 2 + 4 * half) && lane == 0;
        const uint32_t bar_id = 1u + static_cast<uint32_t>(half);
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t acc_empty_local = smem_u32(&ctl->acc_empty[0]);
        const uint32_t stage0 = epi_smem + static_cast<uint32_t>(half * kEpiBufs * kChunkB);
        uint8_t *stage0_ptr = epi_ptr + half * kEpiBufs * kChunkB;
        const int rl = q * 32 + lane;                           // row within the CTA's 128

        // Origin (first row, first column, slice) of chunk c of this half in work unit w.
        // With K splits, D is the partial-sum workspace and unit (b, s) goes to slice
        // b * k_splits + s.  A split tail tile's unit goes to its own tile-sized slice of
        // tmW instead (tail = true; rows and columns relative to the tile).  unit_info's
        // divisions cost hundreds of cycles, so callers evaluate it once per unit.
        auto chunk_origin = [&](const UnitInfo &w, int c, int &x, int &y, int &z, bool &tail) {
            tail = w.tail_slice >= 0;
            const int xr = static_cast<int>(rank) * kBM, yr = half * (BN / 2) + c * kCols;
            x = tail ? xr : w.mt * kTileM + xr;
            y = tail ? yr : w.nt * BN + yr;
            z = tail ? w.tail_slice : w.b * p.k_splits + w.ks;
        };
        // Leader: start the C load of chunk gg (if it exists) into buffer gg % kEpiBufs.
        // The loads run ahead of the chunks being combined, into the next unit; that
        // unit's description is kept between calls.
        uint32_t issued = 0;          // C loads issued: chunks [0, issued)
        int ld_tile = -1;
        UnitInfo ld_w{};
        auto load_c_chunk = [&](uint32_t gg) {
            const int tile = cluster_id + static_cast<int>(gg / kChunks) * num_clusters;
            if (tile >= p.total_tiles)
                return;
            if (tile != ld_tile) {
                ld_w = unit_info(p, tile);
                ld_tile = tile;
            }
            int x, y, z;
            bool tail;
            chunk_origin(ld_w, static_cast<int>(gg % kChunks), x, y, z, tail);
            const uint32_t buf = gg % kEpiBufs;
            const uint32_t bar = smem_u32(&ctl->c_full[half][buf]);
            if (!tail && x < p.m && y < p.n) {
                mbar_arrive_expect_tx(bar, kChunkB);
                tma_load_3d(stage0 + buf * kChunkB, &tmD, bar, x, y, z);
            } else {
                mbar_arrive(bar);       // nothing of this chunk is in the matrix
            }
            issued = gg + 1;
        };
        // With in-kernel TF32 rounding the staging buffers also serve the rounding's
        // transposes between tiles, so C loads stay within a tile (issued once its
        // accumulator is ready) instead of running ahead across tile boundaries.
        if (BETA && !kFuse && half_leader)
            for (uint32_t gg = 0; gg < static_cast<uint32_t>(kAhead); ++gg)
                load_c_chunk(gg);
        uint32_t g = 0;                                         // chunks done by this half
        int it = 0;
        CvWalk walk{};                                          // the half leader's walk
        bool cv_more = kFuse;
        if constexpr (kFuse) {
            if (half_leader)
                walk.start(p, cluster_id);
        }
        for (int t = cluster_id; t < p.total_tiles; t += num_clusters, ++it) {
            const int acc = it % kAccBufs;
            const uint32_t acc_phase = (it / kAccBufs) & 1;
            if constexpr (kFuse) {
                // Round sub-units until this tile's accumulator is ready or the walk is
                // over.  The leader decides (test the barrier, else claim) and tells the
                // half through the shared slot; a sub-unit is counted done once every
                // thread's writes are fenced.
                // The leader's bookkeeping runs while the sub-unit's loads are in flight:
                // the previous sub-unit's done count (`unreported`) and the claim of the
                // next one (`pending`, which must be converted before anything else).
                if (cv_more) {
                    const uint32_t acc_bar = smem_u32(&ctl->acc_full[acc]);
                    uint32_t *tile = reinterpret_cast<uint32_t *>(stage0_ptr);
                    if (half_leader)
                        bulk_wait_group_read<0>();              // no store reads the staging
                    int pending = -3;                           // leader: nothing claimed
                    int unreported = -1;                        // leader: item not yet counted
                    for (;;) {
                        if (half_leader) {
                            int code = pending;
                            if (code == -3)
                                code = mbar_test_wait(acc_bar, acc_phase)
                                           ? -2                 // the accumulator is ready
                                           : (ctl->abort_flag ? -1 : walk.claim(p, num_clusters));
                            ctl->cv_slot[half] = code;
                            pending = -3;
                        }
                        named_barrier_sync(bar_id, 128);
                        const int code = ctl->cv_slot[half];
                        if (code < 0) {
                            cv_more = code == -2;
                            break;
                        }
                        cv_convert<kX3>(p, code >> 6, code & 63, rl, tile, bar_id, [&] {
                            if (half_leader) {
                                if (unreported >= 0)
                                    cv_report(p, unreported);
                                unreported = -1;
                                if (!mbar_test_wait(acc_bar, acc_phase))
                                    pending = ctl->abort_flag ? -1 : walk.claim(p, num_clusters);
                            }
                        });
                        fence_proxy_async_shared();
                        named_barrier_sync(bar_id, 128);
                        if (half_leader)
                            unreported = code >> 6;
                    }
                    if (half_leader && unreported >= 0)
                        cv_report(p, unreported);
                }
            }
            bool ok = wait_bounded<CG>(smem_u32(&ctl->acc_full[acc]), acc_phase, ctl, p,
                                       kErrEpilogue);
            if (named_barrier_or(bar_id, 128, !ok || ctl->abort_flag))
                break;
            tc_fence_after();
            const UnitInfo wt = unit_info(p, t);
            const uint32_t g_end = g + static_cast<uint32_t>(kChunks);
            if constexpr (kFuse && BETA) {
                if (half_leader)
                    for (uint32_t gg = g; gg < g + static_cast<uint32_t>(kAhead) && gg < g_end; ++gg)
                        load_c_chunk(gg);
            }
            bool aborted = false;
#pragma unroll 1
            for (int c = 0; c < kChunks; ++c, ++g) {
                const uint32_t buf = g % kEpiBufs;
                uint8_t *sbuf = stage0_ptr + buf * kChunkB;
                if constexpr (BETA) {
                    ok = wait_bounded<CG>(smem_u32(&ctl->c_full[half][buf]),
                                          (g / kEpiBufs) & 1u, ctl, p, kErrEpilogue);
                    if (named_barrier_or(bar_id, 128, !ok || ctl->abort_flag)) {
                        aborted = true;
                        break;
                    }
                }
                __syncwarp();                                   // tcgen05.ld is warp-collective
                const uint32_t taddr = tmem_base + lane_off +
                                       static_cast<uint32_t>(acc * BN + half * (BN / 2) + c * kCols);
                uint32_t v[kCols];
                if constexpr (kCols == 16) {
                    tmem_ld_32x32b_x16(taddr, v);
                } else {
#pragma unroll
                    for (int h = 0; h < kCols / 32; ++h)
                        tmem_ld_32x32b_x32(taddr + 32 * h,
                                           *reinterpret_cast<uint32_t (*)[32]>(v + 32 * h));
                }
                tmem_ld_wait();
                if (c == kChunks - 1) {
                    // This warp has read its part of the accumulator: report to the MMA CTA.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        const uint32_t bar = acc_empty_local + static_cast<uint32_t>(acc * 8);
                        mbar_arrive_cluster(CG == 2 ? mapa_shared(bar, 0) : bar);
                    }
                }
                int cx, cy, cz;
                bool tail_unit;
                chunk_origin(wt, c, cx, cy, cz, tail_unit);
                // A TMA store writes the last row run of a column in whole 16-byte units,
                // which would touch rows >= m inside the ldc padding: a chunk that crosses
                // row m at a non-16-byte boundary is stored by the threads instead.  (Tail
                // partial sums go to whole tile-sized slices and never need that.)
                const bool thread_store = !tail_unit && cx + kBM > p.m &&
                                          (static_cast<int64_t>(p.m) * kOutBytes) % 16 != 0;
                float r[kCols];
                if (OUT == kOutF32 && tail_unit) {
                    // the raw FP32 accumulator; the tail reduction applies alpha and beta
#pragma unroll
                    for (int j = 0; j < kCols; ++j)
                        r[j] = __uint_as_float(v[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < kCols; ++j) {
                        r[j] = p.alpha * __uint_as_float(v[j]);
                        if constexpr (BETA)
                            r[j] = fmaf(p.beta, load_smem<OUT>(sbuf, j * kBM + rl), r[j]);
                    }
                }
                if (!thread_store) {
                    if constexpr (OUT == kOutF32) {
#pragma unroll
                        for (int j = 0; j < kCols; ++j)
                            store_smem<OUT>(sbuf, j * kBM + rl, r[j]);
                    } else {
#pragma unroll
                        for (int j = 0; j < kCols; j += 2)
                            store_smem_pair<OUT>(sbuf, j * kBM + rl, kBM, r[j], r[j + 1]);
                    }
                } else if (cx + rl < p.m) {
                    const int64_t base_idx = static_cast<int64_t>(cz) * p.strideC + cx + rl;
#pragma unroll
                    for (int j = 0; j < kCols; ++j)
                        if (cy + j < p.n)
                            store_out<OUT>(p.D, base_idx + static_cast<int64_t>(cy + j) * p.ldc,
                                           r[j]);
                }
                fence_proxy_async_shared();
                named_barrier_sync(bar_id, 128);               // the block is complete
                if (half_leader) {
                    if (tail_unit)
                        tma_store_3d(&tmW, stage0 + buf * kChunkB, cx, cy, cz);
                    else if (!thread_store && cx < p.m && cy < p.n)
                        tma_store_3d(&tmD, stage0 + buf * kChunkB, cx, cy, cz);
                    bulk_commit_group();
                    // The buffer of chunk g + 1 (no C) or g + kAhead (C) was last stored
                    // from by chunk g + 1 - kEpiBufs: allow only this chunk's store pending.
                    bulk_wait_group_read<1>();
                    if constexpr (BETA) {
                        if (!kFuse || g + kAhead < g_end)
                            load_c_chunk(g + kAhead);
                    }
                }
                named_barrier_sync(bar_id, 128);               // the next buffer is free
            }
            if (aborted)
                break;
        }
        if (half_leader) {
            // Aborted with C loads in flight: let them land (bounded).
            for (uint32_t gg = g; gg < issued; ++gg)
                wait_bounded<CG>(smem_u32(&ctl->c_full[half][gg % kEpiBufs]),
                                 (gg / kEpiBufs) & 1u, ctl, p, kErrDrain, false);
            bulk_wait_group_all();
        }
    }

    tc_fence_before();
    if constexpr (CG == 2)
        cluster_sync_all();
    else
        __syncthreads();
    if (ctl->abort_flag && warp == 0 && lane == 0) {
        // Aborted: let every load already issued land before the CTA leaves.  The
        // leader waits on its stage barriers (which count both CTAs' bytes); both CTAs
        // then give straggling copies a further 20 us.
        if (leader)
            for (int s = 0; s < kStages; ++s)
                if (issued_mask & (1u << s))
                    wait_bounded<CG>(smem_u32(&ctl->full[s]), (issued_parity >> s) & 1u, ctl, p,
                                     kErrDrain, false);
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 20000ull) {
        }
    }
    if constexpr (CG == 2)
        cluster_sync_all();
    else
        __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if constexpr (CG == 2)
            tmem_dealloc_pair(tmem_base, kTmemCols);
        else
            tmem_dealloc(tmem_base, kTmemCols);
    }
    if (p.clk && threadIdx.x == 0) {
        atomicAdd(p.clk, static_cast<unsigned long long>(clock64()) - clk0);
        atomicAdd(p.clk + 1, globaltimer_ns() - ns0);
    }
}

template <int OUT>
__global__ void tcg_scale_kernel(void *D, const void *C, int m, int n, int64_t ldc,
                                 int64_t strideC, int batch, float beta)
{
    const int64_t per = static_cast<int64_t>(m) * n;
    const int64_t total = per * batch;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t b = e / per;
        const int64_t r = e - b * per;
        const int64_t j = r / m;
        const int64_t i = r - j * m;
        const int64_t idx = b * strideC + i + j * ldc;
        const float v = (beta == 0.0f) ? 0.0f : beta * load_c<OUT>(C, idx);
        store_out<OUT>(D, idx, v);
    }
}

// Split-K reduction: D = alpha * sum_s W_s + beta * C, the partial sums W_s (FP32, one
// slice per K range of every batch entry) added in range order in FP32, then the same
// epilogue arithmetic as the GEMM kernel (alpha * acc, fma with beta * C, one rounding to
// the output type).  A block takes one column of one batch entry at a time (grid-stride
// over the batch x n columns), its threads the rows: every slice and C/D are read and
// written along contiguous rows, and the index arithmetic is done once per column.
template <int OUT>
__global__ void __launch_bounds__(256) tcg_splitk_reduce_kernel(const float *__restrict__ W,
                                                                int64_t ldw, int splits, int m,
                                                                int n, int batch, float alpha,
                                                                float beta, void *D, int64_t ldc,
                                                                int64_t strideC)
{
    griddep_wait();
    const int64_t slice = ldw * n;
    const int64_t cols = static_cast<int64_t>(batch) * n;
    for (int64_t bj = blockIdx.x; bj < cols; bj += gridDim.x) {
        const int64_t b = bj / n;
        const int64_t j = bj - b * n;
        const float *wcol = W + b * splits * slice + j * ldw;
        const int64_t dcol = b * strideC + j * ldc;
        for (int i = threadIdx.x; i < m; i += blockDim.x) {
            float acc = wcol[i];
            for (int s = 1; s < splits; ++s)
                acc = __fadd_rn(acc, wcol[s * slice + i]);
            float v = __fmul_rn(alpha, acc);
            if (beta != 0.0f)
                v = __fmaf_rn(beta, load_c<OUT>(D, dcol + i), v);
            store_out<OUT>(D, dcol + i, v);
        }
    }
    griddep_launch_dependents();
}

// Tail reduction (FP32 output only): for each split tail tile r (tiles full_units + r),
// D = alpha * (W[r*S] + W[r*S + 1] + ... in that order, FP32) + beta * C over the tile's
// elements inside the matrix.  W slices are tile-sized (tile_m x 256 FP32, leading
// dimension tile_m).  A block takes 16 columns of one tail tile at a time (grid-stride
// over tail tiles x 16 column groups; the tile's position is worked out once per group),
// its threads the rows; every thread keeps 16 x S loads in flight.
constexpr int kTailCols = 16;
__global__ void __launch_bounds__(256) tcg_tail_reduce_kernel(const float *__restrict__ W,
                                                              int tail_tiles, int tile_m,
                                                              const GemmArgs p)
{
    griddep_wait();
    constexpr int kGroups = kBN / kTailCols;
    const int64_t per_tile = static_cast<int64_t>(tile_m) * kBN;
    const int S = p.tail_splits;
    const int groups = tail_tiles * kGroups;
    for (int rg = blockIdx.x; rg < groups; rg += gridDim.x) {
        const int r = rg / kGroups;
        const int j0l = (rg - r * kGroups) * kTailCols;
        int b, mt, nt;
        raster(p, p.full_units + r, b, mt, nt);
        const int i0 = mt * tile_m, jb = nt * kBN + j0l;
        const float *wt = W + static_cast<int64_t>(r) * S * per_tile + static_cast<int64_t>(j0l) * tile_m;
        for (int il = threadIdx.x; il < tile_m && i0 + il < p.m; il += blockDim.x) {
            float acc[kTailCols];
#pragma unroll
            for (int jj = 0; jj < kTailCols; ++jj)
                acc[jj] = wt[jj * tile_m + il];
            for (int s = 1; s < S; ++s) {
                const float *ws = wt + s * per_tile;
#pragma unroll
                for (int jj = 0; jj < kTailCols; ++jj)
                    acc[jj] = __fadd_rn(acc[jj], ws[jj * tile_m + il]);
            }
            const int64_t row = static_cast<int64_t>(b) * p.strideC + i0 + il;
#pragma unroll
            for (int jj = 0; jj < kTailCols; ++jj) {
                if (jb + jj >= p.n)
                    break;
                const int64_t idx = row + static_cast<int64_t>(jb + jj) * p.ldc;
                float v = __fmul_rn(p.alpha, acc[jj]);
                if (p.beta != 0.0f)
                    v = __fmaf_rn(p.beta, static_cast<const float *>(p.C)[idx], v);
                static_cast<float *>(p.D)[idx] = v;
            }
        }
    }
    griddep_launch_dependents();
}

// out[b][r][p] = tf32(op element (r, p)) with rows r < rows (the M or N extent) and K
// contiguous (ld_out elements per row).  The input element (r, p) sits at
// in[b*stride_in + p + r*ld] (K-major) or in[b*stride_in + r + p*ld] (M/N-major).
// 32x32 tiles through shared memory so both sides stay coalesced.
__global__ void __launch_bounds__(256) tcg_tf32_pack_kernel(const uint32_t *__restrict__ in,
                                                            int64_t ld, int64_t stride_in,
                                                            int in_kmajor, int rows, int k,
                                                            int batch, uint32_t *__restrict__ out,
                                                            int64_t ld_out, int64_t stride_out)
{
    __shared__ uint32_t tile[32][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8
    const int64_t tr = (rows + 31) / 32, tk = (k + 31) / 32;
    const int64_t total = tr * tk * batch;
    for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
        const int64_t b = t / (tr * tk);
        const int64_t rem = t - b * tr * tk;
        const int r0 = static_cast<int>(rem / tk) * 32;
        const int p0 = static_cast<int>(rem % tk) * 32;
        const uint32_t *src = in + b * stride_in;
        __syncthreads();
        if (in_kmajor) {
            for (int i = ty; i < 32; i += 8) {
                const int r = r0 + i, pp = p0 + tx;
                tile[i][tx] = (r < rows && pp < k) ? src[pp + static_cast<int64_t>(r) * ld] : 0u;
            }
        } else {
            for (int i = ty; i < 32; i += 8) {
                const int pp = p0 + i, r = r0 + tx;
                tile[tx][i] = (r < rows && pp < k) ? src[r + static_cast<int64_t>(pp) * ld] : 0u;
            }
        }
        __syncthreads();
        uint32_t *dst = out + b * stride_out;
        for (int i = ty; i < 32; i += 8) {
            const int r = r0 + i, pp = p0 + tx;
            if (r < rows && pp < k)
                dst[pp + static_cast<int64_t>(r) * ld_out] = tf32_rne_bits(tile[i][tx]);
        }
    }
}

typedef void (*GemmKernelFn)(const CUtensorMap, const CUtensorMap, const CUtensorMap,
                             const CUtensorMap, const CUtensorMap, const CUtensorMap,
                             const GemmArgs);

template <int CG, int CBUF>
static GemmKernelFn gemm_fn_cg(int out_kind, int kind)
{
    if (kind == kKindTF32)   // TF32 inputs always produce FP32 output
        return tcg_gemm_kernel<kOutF32, CG, kKindTF32, CBUF, kBN>;
    if (kind == kKindTF32x3)
        return tcg_gemm_kernel<kOutF32, CG, kKindTF32x3, CBUF, kBN>;
    if (kind == kKindTF32R)
        return tcg_gemm_kernel<kOutF32, CG, kKindTF32R, CBUF, kBN>;
    if (kind == kKindTF32x3R)
        return tcg_gemm_kernel<kOutF32, CG, kKindTF32x3R, CBUF, kBN>;
    if (kind == kKindF8) {
        switch (out_kind) {
        case kOutF32: return tcg_gemm_kernel<kOutF32, CG, kKindF8, CBUF, kBN>;
        case kOutF16: return tcg_gemm_kernel<kOutF16, CG, kKindF8, CBUF, kBN>;
        default: return tcg_gemm_kernel<kOutBF16, CG, kKindF8, CBUF, kBN>;
        }
    }
    switch (out_kind) {
    case kOutF32: return tcg_gemm_kernel<kOutF32, CG, kKindF16, CBUF, kBN>;
    case kOutF16: return tcg_gemm_kernel<kOutF16, CG, kKindF16, CBUF, kBN>;
    default: return tcg_gemm_kernel<kOutBF16, CG, kKindF16, CBUF, kBN>;
    }
}

// Narrow tiles (kBNNarrow): SM pairs with FP16/BF16 inputs only.
template <int CBUF>
static GemmKernelFn gemm_fn_narrow(int out_kind)
{
    switch (out_kind) {
    case kOutF32: return tcg_gemm_kernel<kOutF32, 2, kKindF16, CBUF, kBNNarrow>;
    case kOutF16: return tcg_gemm_kernel<kOutF16, 2, kKindF16, CBUF, kBNNarrow>;
    default: return tcg_gemm_kernel<kOutBF16, 2, kKindF16, CBUF, kBNNarrow>;
    }
}

bool gemm_has_narrow(int cta_group, int kind)
{
    return cta_group == 2 && kind == kKindF16;
}

// c_bufs: 0 (beta == 0), 2 or 4 (C staging buffers per epilogue half; 4 only for pairs).
static GemmKernelFn gemm_fn(int out_kind, int cta_group, int kind, int c_bufs, int bn = kBN)
{
    if (bn == kBNNarrow && gemm_has_narrow(cta_group, kind))
        return c_bufs == 4 ? gemm_fn_narrow<4>(out_kind)
                           : (c_bufs ? gemm_fn_narrow<2>(out_kind) : gemm_fn_narrow<0>(out_kind));
    if (cta_group == 2) {
        if (c_bufs == 4)
            return gemm_fn_cg<2, 4>(out_kind, kind);
        return c_bufs ? gemm_fn_cg<2, 2>(out_kind, kind) : gemm_fn_cg<2, 0>(out_kind, kind);
    }
    return c_bufs ? gemm_fn_cg<1, 2>(out_kind, kind) : gemm_fn_cg<1, 0>(out_kind, kind);
}

static cudaError_t prepare(GemmKernelFn fn)
{
    // cudaFuncSetAttribute is cheap; doing it per launch keeps the code free of
    // per-device caches.
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

int gemm_max_resident_ctas(int cta_group, int num_sms)
{
    GemmKernelFn fn = gemm_fn(kOutF32, cta_group, kKindF16, 0);
    if (prepare(fn) != cudaSuccess) {
        cudaGetLastError();
        return num_sms / cta_group * cta_group;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(num_sms / cta_group * cta_group, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cta_group;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) != cudaSuccess || clusters <= 0) {
        cudaGetLastError();
        return num_sms / cta_group * cta_group;
    }
    return clusters * cta_group;
}

// K-major operand (K contiguous, `ld` elements per row of op, `rows` = K, `cols` = M or
// N): out[b][c][r] = tf32(in[b][c][r]), 4 elements (16 bytes) per access.  With out_lo
// the two-word split is written instead: out = hi, out_lo = lo (same layout).  ld, ld_out
// and the strides are multiples of 4 elements and the pointers 16-byte aligned, so r runs
// up to round_up(rows, 4), which stays inside every column's storage.
__global__ void __launch_bounds__(256) tcg_tf32_round_kernel(const uint4 *__restrict__ in,
                                                             int64_t ld4, int64_t stride_in4,
                                                             int rows4, int cols, int batch,
                                                             uint4 *__restrict__ out,
                                                             int64_t ld_out4, int64_t stride_out4,
                                                             uint4 *__restrict__ out_lo)
{
    griddep_wait();
    for (int b = blockIdx.z; b < batch; b += gridDim.z)
        for (int c = blockIdx.y; c < cols; c += gridDim.y) {
            const uint4 *src = in + b * stride_in4 + static_cast<int64_t>(c) * ld4;
            const int64_t o = b * stride_out4 + static_cast<int64_t>(c) * ld_out4;
            for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < rows4;
                 r += gridDim.x * blockDim.x) {
                uint4 v = src[r];
                if (out_lo) {
                    uint4 lo;
                    tf32_split_bits(v.x, v.x, lo.x);
                    tf32_split_bits(v.y, v.y, lo.y);
                    tf32_split_bits(v.z, v.z, lo.z);
                    tf32_split_bits(v.w, v.w, lo.w);
                    out_lo[o + r] = lo;
                } else {
                    v.x = tf32_rne_bits(v.x);
                    v.y = tf32_rne_bits(v.y);
                    v.z = tf32_rne_bits(v.z);
                    v.w = tf32_rne_bits(v.w);
                }
                out[o + r] = v;
            }
        }
    griddep_launch_dependents();
}

// M/N-major operand: element (r, p) (r < rows along M or N, p < k along K) at
// in[b*stride_in + r + p*ld]; writes the K-major copy out[b*stride_out + p + r*ld_out],
// rounded, for p < round_up(k, 4) (zeros past k).  64 x 64 tiles through shared memory
// with 16-byte global accesses on both sides: 16 threads read one K row's 64 elements
// (four per thread) and 16 threads write one output row's 64; the 65-word row pitch
// keeps both shared-memory phases at two-way bank conflicts at most.  ld, ld_out and the
// strides are multiples of 4 elements and the pointers 16-byte aligned, so the four
// elements read past `rows` stay inside the column's storage (ld >= round_up(rows, 4)).
__global__ void __launch_bounds__(256) tcg_tf32_transpose_round_kernel(
    const uint32_t *__restrict__ in, int64_t ld, int64_t stride_in, int rows, int k, int batch,
    uint32_t *__restrict__ out, int64_t ld_out, int64_t stride_out, uint32_t *__restrict__ out_lo)
{
    __shared__ uint32_t tile[64][65];                 // [p][r]
    griddep_wait();
    const int c = threadIdx.x & 15, w = threadIdx.x >> 4;
    const int r_tiles = (rows + 63) / 64, p_tiles = (k + 63) / 64;
    for (int b = blockIdx.z; b < batch; b += gridDim.z)
        for (int pt = blockIdx.y; pt < p_tiles; pt += gridDim.y)
            for (int rt = blockIdx.x; rt < r_tiles; rt += gridDim.x) {
                const int r0 = rt * 64, p0 = pt * 64;
                const uint32_t *src = in + b * stride_in;
                __syncthreads();
#pragma unroll
                for (int j = 0; j < 4; ++j) {               // K rows p0 + w + 16 j
                    const int pl = w + 16 * j, pp = p0 + pl, r = r0 + 4 * c;
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (pp < k && r < rows)
                        v = *reinterpret_cast<const uint4 *>(src + r +
                                                             static_cast<int64_t>(pp) * ld);
                    tile[pl][4 * c] = v.x;
                    tile[pl][4 * c + 1] = v.y;
                    tile[pl][4 * c + 2] = v.z;
                    tile[pl][4 * c + 3] = v.w;
                }
                __syncthreads();
#pragma unroll
                for (int j = 0; j < 4; ++j) {               // output rows r0 + w + 16 j
                    const int rl = w + 16 * j, r = r0 + rl, pp = p0 + 4 * c;
                    if (r >= rows || pp >= k)
                        continue;
                    const uint32_t x[4] = {tile[4 * c][rl], tile[4 * c + 1][rl],
                                           tile[4 * c + 2][rl], tile[4 * c + 3][rl]};
                    const int64_t o = b * stride_out + pp + static_cast<int64_t>(r) * ld_out;
                    uint4 hi, lo;
                    if (out_lo) {
                        tf32_split_bits(x[0], hi.x, lo.x);
                        tf32_split_bits(x[1], hi.y, lo.y);
                        tf32_split_bits(x[2], hi.z, lo.z);
                        tf32_split_bits(x[3], hi.w, lo.w);
                        *reinterpret_cast<uint4 *>(out_lo + o) = lo;
                    } else {
                        hi = make_uint4(tf32_rne_bits(x[0]), tf32_rne_bits(x[1]),
                                        tf32_rne_bits(x[2]), tf32_rne_bits(x[3]));
                    }
                    *reinterpret_cast<uint4 *>(out + o) = hi;
                }
            }
    griddep_launch_dependents();
}

static inline unsigned clamp_grid(int64_t v, int64_t cap)
{
    return static_cast<unsigned>(v < 1 ? 1 : (v > cap ? cap : v));
}

// Launch with programmatic stream serialization (the kernel waits in griddepcontrol.wait
// before it reads anything and lets its own dependents launch at its end), so a chain
// of the library's kernels on one stream hides each launch behind the previous kernel.
template <typename... Params, typename... Args>
static cudaError_t launch_chained(void (*kernel)(Params...), dim3 grid, dim3 block,
                                  cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_tf32_round(const void *in, int64_t ld, int64_t stride_in, int64_t rows,
                              int64_t cols, int64_t batch, void *out, int64_t ld_out,
                              int64_t stride_out, void *out_lo, cudaStream_t s)
{
    const int64_t rows4 = (rows + 3) / 4;
    const dim3 g(clamp_grid((rows4 + 255) / 256, 1 << 16), clamp_grid(cols, 65535),
                 clamp_grid(batch, 65535));
    return launch_chained(tcg_tf32_round_kernel, g, dim3(256), s,
                          static_cast<const uint4 *>(in), ld / 4, stride_in / 4,
                          static_cast<int>(rows4), static_cast<int>(cols),
                          static_cast<int>(batch), static_cast<uint4 *>(out), ld_out / 4,
                          stride_out / 4, static_cast<uint4 *>(out_lo));
}

cudaError_t launch_tf32_transpose_round(const void *in, int64_t ld, int64_t stride_in,
                                        int64_t rows, int64_t k, int64_t batch, void *out,
                                        int64_t ld_out, int64_t stride_out, void *out_lo,
                                        cudaStream_t s)
{
    const dim3 g(clamp_grid((rows + 63) / 64, (int64_t(1) << 31) - 1),
                 clamp_grid((k + 63) / 64, 65535), clamp_grid(batch, 65535));
    return launch_chained(tcg_tf32_transpose_round_kernel, g, dim3(256), s,
                          static_cast<const uint32_t *>(in), ld, stride_in,
                          static_cast<int>(rows), static_cast<int>(k), static_cast<int>(batch),
                          static_cast<uint32_t *>(out), ld_out, stride_out,
                          static_cast<uint32_t *>(out_lo));
}

cudaError_t launch_gemm(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmD,
                        const CUtensorMap &tmW, const GemmArgs &a, int out_kind, int cta_group,
                        int bn, int grid, cudaStream_t s, const CUtensorMap *tmA2,
                        const CUtensorMap *tmB2)
{
    const bool two_words = a.kind == kKindTF32x3 || a.kind == kKindTF32x3R;
    if (two_words != (tmA2 != nullptr && tmB2 != nullptr))
        return cudaErrorInvalidValue;
    if (bn != kBN && !(bn == kBNNarrow && gemm_has_narrow(cta_group, a.kind)))
        return cudaErrorInvalidValue;
    GemmKernelFn fn = gemm_fn(out_kind, cta_group, a.kind, a.c_bufs, bn);
    cudaError_t e = prepare(fn);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cta_group;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // Programmatic dependent launch: the kernel may start while the previous kernel on the
    // stream finishes (it waits in griddepcontrol.wait before any global access).
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, fn, tmA, tmB, tmD, tmW, tmA2 ? *tmA2 : tmA, tmB2 ? *tmB2 : tmB, a);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

cudaError_t launch_scale(void *D, const void *C, int m, int n, int64_t ldc, int64_t strideC,
                         int batch, float beta, int out_kind, int grid, cudaStream_t s)
{
    switch (out_kind) {
    case kOutF32: tcg_scale_kernel<kOutF32><<<grid, 256, 0, s>>>(D, C, m, n, ldc, strideC, batch, beta); break;
    case kOutF16: tcg_scale_kernel<kOutF16><<<grid, 256, 0, s>>>(D, C, m, n, ldc, strideC, batch, beta); break;
    default: tcg_scale_kernel<kOutBF16><<<grid, 256, 0, s>>>(D, C, m, n, ldc, strideC, batch, beta); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_splitk_reduce(const float *W, int64_t ldw, int splits, int m, int n, int batch,
                                 float alpha, float beta, void *D, int64_t ldc, int64_t strideC,
                                 int out_kind, int grid, cudaStream_t s)
{
    auto fn = out_kind == kOutF32 ? tcg_splitk_reduce_kernel<kOutF32>
            : (out_kind == kOutF16 ? tcg_splitk_reduce_kernel<kOutF16>
                                   : tcg_splitk_reduce_kernel<kOutBF16>);
    return launch_chained(fn, dim3(grid), dim3(256), s, W, ldw, splits, m, n, batch, alpha,
                          beta, D, ldc, strideC);
}

cudaError_t launch_tail_reduce(const float *W, int tail_tiles, int tile_m, const GemmArgs &a,
                               int grid, cudaStream_t s)
{
    return launch_chained(tcg_tail_reduce_kernel, dim3(grid), dim3(256), s, W, tail_tiles,
                          tile_m, a);
}

cudaError_t launch_tf32_pack(const void *in, int64_t ld, int64_t stride_in, int in_kmajor,
                             int rows, int k, int batch, void *out, int64_t ld_out,
                             int64_t stride_out, int grid, cudaStream_t s)
{
    tcg_tf32_pack_kernel<<<grid, 256, 0, s>>>(static_cast<const uint32_t *>(in), ld, stride_in,
                                              in_kmajor, rows, k, batch,
                                              static_cast<uint32_t *>(out), ld_out, stride_out);
    return cudaGetLastError();
}

}  // namespace tcg
