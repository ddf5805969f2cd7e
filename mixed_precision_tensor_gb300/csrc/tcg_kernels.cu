// tcg_kernels.cu -- device code of libtcg (sm_103a).
//
// tcg_gemm_kernel: persistent, warp-specialised tensor-core GEMM
//     D = alpha * op(A) * op(B) + beta * C
// ("Programming Tensor Cores in CUDA 9", sections "什么是张量核?" and "CUDA 9.0 中
// 张量核的编程访问": exact products, FP32 accumulation, alpha/beta applied to the
// accumulator elementwise; "CUDA Handbook, 17.5 Tensor Cores": one MMA instruction
// is a rank-K slab of the outer-product sum over k).
//
//   warp 0 (one lane)   TMA producer: 128x(128 B) A tile and 256x(128 B) B tile per
//                        stage into a 4-deep ring of 128-byte-swizzled shared memory;
//                        out-of-range rows/columns/K are zero-filled by TMA, which
//                        makes ragged m, n, k exact.
//   warp 1 (one lane)   MMA issuer: tcgen05.mma (M=128, N=256, K=16 for FP16/BF16,
//                        K=8 for TF32) into a TMEM accumulator; two accumulators
//                        (2 x 256 columns) so the epilogue of tile t overlaps the
//                        main loop of tile t+1.  The page's diagnosis -- a tensor-core
//                        kernel that stalls waiting for the next slab ("CUDA Handbook,
//                        17.5", after Listing 17-5) -- is what the ring and the
//                        separate producer remove.
//   warps 2-5           epilogue: tcgen05.ld TMEM -> registers, alpha*acc + beta*C in
//                        FP32, round to the output type (nearest even), coalesced
//                        column-major stores (a warp writes 32 consecutive rows).
//
// Every wait is bounded (globaltimer): a wait that runs out sets a bit in the device
// error word and a shared abort flag, every role stops, in-flight copies and MMAs are
// drained, TMEM is freed and the kernel returns.  No trap, no unbounded spin.
//
// tcg_scale_kernel: D = beta * C (k == 0 or alpha == 0, A and B not read).
// tcg_tf32_pack_kernel: FP32 -> TF32 (round to nearest even) into a K-major copy.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tcg_internal.h"
#include "tcg_ptx.cuh"

namespace tcg {

struct SmemCtl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full[kAccBufs];
    uint64_t acc_empty[kAccBufs];
    uint64_t drain;
    uint32_t tmem_base;
    volatile int abort_flag;
};
static_assert(sizeof(SmemCtl) <= kBarrierBytes, "barrier area too small");

// Bounded wait on an mbarrier phase.  Returns false if the kernel was aborted or the
// limit ran out (then the error bit is recorded and the abort flag raised).
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
            ctl->abort_flag = 1;
            atomicOr(p.err, err_bit);
            return false;
        }
    }
}

__device__ __forceinline__ void tile_coords(const GemmArgs &p, int t, int &b, int &mt, int &nt)
{
    const int per_batch = p.num_m_tiles * p.num_n_tiles;
    b = t / per_batch;
    const int r = t - b * per_batch;
    const int span = p.group_m * p.num_n_tiles;
    const int g = r / span;
    const int first_m = g * p.group_m;
    const int gsize = min(p.num_m_tiles - first_m, p.group_m);
    const int in_g = r - g * span;
    mt = first_m + in_g % gsize;
    nt = in_g / gsize;
}

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
__device__ __forceinline__ float load_c(const void *C, int64_t idx)
{
    if constexpr (OUT == kOutF32)
        return static_cast<const float *>(C)[idx];
    else if constexpr (OUT == kOutF16)
        return __half2float(static_cast<const __half *>(C)[idx]);
    else
        return __bfloat162float(static_cast<const __nv_bfloat16 *>(C)[idx]);
}

template <int OUT>
__global__ void __launch_bounds__(kThreads, 1)
    tcg_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB, const GemmArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms.
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base = (raw_u32 + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw_u32);
    const uint32_t a_smem = base;
    const uint32_t b_smem = base + kStages * kABytes;
    SmemCtl *ctl = reinterpret_cast<SmemCtl *>(base_ptr + kStages * kStageBytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int a = 0; a < kAccBufs; ++a) {
            mbar_init(smem_u32(&ctl->acc_full[a]), 1);
            mbar_init(smem_u32(&ctl->acc_empty[a]), kEpiWarps);
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;

    // Byte offsets of successive K slices (one MMA each) inside a stage, and the
    // descriptor strides, per operand majorness.
    const int esize = p.is_tf32 ? 4 : 2;
    const uint32_t k_mma = 32u / esize;                       // K per MMA instruction
    const uint32_t chunk_bytes = static_cast<uint32_t>(p.k_per_block) * kRowBytes;
    const uint32_t a_kstep = p.a_kmajor ? 32u : k_mma * kRowBytes;
    const uint32_t b_kstep = p.b_kmajor ? 32u : k_mma * kRowBytes;
    const uint32_t a_lbo = p.a_kmajor ? 16u : chunk_bytes;
    const uint32_t b_lbo = p.b_kmajor ? 16u : chunk_bytes;
    constexpr uint32_t kSbo = 8 * kRowBytes;                  // 8-row group stride
    const int mmas_per_stage = kRowBytes / 32;                // 4
    uint32_t issued_mask = 0, issued_parity = 0;              // producer: loads issued per stage

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ producer
            int stage = 0;
            uint32_t phase = 0;
            bool skip_once = p.fault_inject != 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x) {
                int b, mt, nt;
                tile_coords(p, t, b, mt, nt);
                const int m0 = mt * kBM, n0 = nt * kBN;
                const int za = p.a_bcast ? 0 : b, zb = p.b_bcast ? 0 : b;
                for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                    const uint32_t fb = smem_u32(&ctl->full[stage]);
                    if (!wait_bounded(smem_u32(&ctl->empty[stage]), phase ^ 1u, ctl, p,
                                      kErrProducer)) {
                        ok = false;
                        break;
                    }
                    if (skip_once) {
                        skip_once = false;  // test hook: this stage is never filled
                    } else {
                        mbar_arrive_expect_tx(fb, kStageBytes);
                        const uint32_t sa = a_smem + stage * kABytes;
                        const uint32_t sb = b_smem + stage * kBBytes;
                        const int k0 = kb * p.k_per_block;
                        if (p.a_kmajor) {
                            tma_load_3d(sa, &tmA, fb, k0, m0, za);
                        } else {
                            for (int h = 0; h < kBM / p.mn_box; ++h)
                                tma_load_3d(sa + h * chunk_bytes, &tmA, fb, m0 + h * p.mn_box, k0,
                                            za);
                        }
                        if (p.b_kmajor) {
                            tma_load_3d(sb, &tmB, fb, k0, n0, zb);
                        } else {
                            for (int h = 0; h < kBN / p.mn_box; ++h)
                                tma_load_3d(sb + h * chunk_bytes, &tmB, fb, n0 + h * p.mn_box, k0,
                                            zb);
                        }
                        issued_mask |= 1u << stage;
                        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ----------------------------------------------------------- MMA issue
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x, ++it) {
                const int acc = it & 1;
                const uint32_t acc_phase = (it >> 1) & 1;
                if (!wait_bounded(smem_u32(&ctl->acc_empty[acc]), acc_phase ^ 1u, ctl, p,
                                  kErrMmaAcc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
                for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                    if (!wait_bounded(smem_u32(&ctl->full[stage]), phase, ctl, p, kErrMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = a_smem + stage * kABytes;
                    const uint32_t sb = b_smem + stage * kBBytes;
                    for (int kk = 0; kk < mmas_per_stage; ++kk) {
                        const uint64_t ad = smem_desc_sw128(sa + kk * a_kstep, a_lbo, kSbo);
                        const uint64_t bd = smem_desc_sw128(sb + kk * b_kstep, b_lbo, kSbo);
                        const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
                        if (p.is_tf32)
                            mma_tf32(d_tmem, ad, bd, p.idesc, accum);
                        else
                            mma_f16(d_tmem, ad, bd, p.idesc, accum);
                    }
                    mma_commit(smem_u32(&ctl->empty[stage]));  // stage free once read
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                mma_commit(smem_u32(&ctl->acc_full[acc]));     // accumulator ready
            }
            // Every MMA issued so far must be complete before TMEM is released.
            mma_commit(smem_u32(&ctl->drain));
            wait_bounded(smem_u32(&ctl->drain), 0, ctl, p, kErrDrain, false);
        }
    } else {
        // -------------------------------------------------------------- epilogue
        const int q = warp & 3;                       // TMEM lane quarter of this warp
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        int it = 0;
        for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++it) {
            const int acc = it & 1;
            const uint32_t acc_phase = (it >> 1) & 1;
            bool ok = wait_bounded(smem_u32(&ctl->acc_full[acc]), acc_phase, ctl, p, kErrEpilogue);
            if (!__all_sync(0xffffffffu, ok))
                break;
            tc_fence_after();
            int b, mt, nt;
            tile_coords(p, t, b, mt, nt);
            const int row = mt * kBM + q * 32 + lane;
            const bool row_ok = row < p.m;
            const int64_t boff = static_cast<int64_t>(b) * p.strideC;
            for (int c = 0; c < kBN / 32; ++c) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem_base + lane_off + static_cast<uint32_t>(acc * kBN + c * 32),
                                   v);
                tmem_ld_wait();
                if (c == kBN / 32 - 1) {
                    // Accumulator fully read: hand it back to the MMA warp.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(smem_u32(&ctl->acc_empty[acc]));
                }
                const int col0 = nt * kBN + c * 32;
                if (row_ok) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int col = col0 + j;
                        if (col < p.n) {
                            const int64_t idx = boff + row + static_cast<int64_t>(col) * p.ldc;
                            float r = p.alpha * __uint_as_float(v[j]);
                            if (p.beta != 0.0f)
                                r = fmaf(p.beta, load_c<OUT>(p.C, idx), r);
                            store_out<OUT>(p.D, idx, r);
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (ctl->abort_flag && warp == 0 && lane == 0) {
        // Aborted: let every load already issued land before the CTA leaves.
        for (int s = 0; s < kStages; ++s)
            if (issued_mask & (1u << s))
                wait_bounded(smem_u32(&ctl->full[s]), (issued_parity >> s) & 1u, ctl, p,
                             kErrDrain, false);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
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

cudaError_t launch_gemm(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmArgs &a,
                        int out_kind, int grid, cudaStream_t s)
{
    static bool attr_set[3] = {false, false, false};
    void (*fn)(const CUtensorMap, const CUtensorMap, const GemmArgs) = nullptr;
    switch (out_kind) {
    case kOutF32: fn = tcg_gemm_kernel<kOutF32>; break;
    case kOutF16: fn = tcg_gemm_kernel<kOutF16>; break;
    default: fn = tcg_gemm_kernel<kOutBF16>; break;
    }
    if (!attr_set[out_kind]) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemBytes);
        if (e != cudaSuccess)
            return e;
        attr_set[out_kind] = true;
    }
    fn<<<grid, kThreads, kSmemBytes, s>>>(tmA, tmB, a);
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
