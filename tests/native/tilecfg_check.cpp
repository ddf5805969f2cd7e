/*
 * Host-side check of the GEMM kernel's shared-memory plan (tcg::TileCfg and the epilogue
 * chunk rule in tcg_internal.h) for every variant the library instantiates: the operand
 * ring and the epilogue staging fill the data area exactly, both are multiples of the
 * 1 KiB swizzle atom, the ring keeps at least two stages for every MMA kind (the
 * two-word TF32 kind carries four operand tiles per stage), an epilogue chunk is a whole
 * TMA box (at most 256 columns, a whole number of chunks per half tile), and with C read
 * at least one C chunk is in flight.  Test code only.
 */
#include <cstdint>

#include "tcg_internal.h"

namespace {

template <int CG, int CBUF, int BN, int OUT_BYTES>
int check_one()
{
    using namespace tcg;
    constexpr int chunk = epi_chunk_bytes(OUT_BYTES, CBUF);
    using Cfg = TileCfg<CG, CBUF, BN, chunk>;
    int bad = 0;
    bad += (Cfg::kRingBytes + Cfg::kEpiBytes != kDataBytes);
    bad += (Cfg::kRingBytes % 1024 != 0) + (Cfg::kEpiBytes % 1024 != 0);
    bad += (Cfg::kStages < 2);                                  // one word per operand
    bad += (Cfg::kRingBytes / (2 * Cfg::kStageBytes) < 2);      // two words (3xTF32)
    bad += (kSmemBytes > 227 * 1024);
    constexpr int cols = epi_cols(OUT_BYTES, CBUF);
    bad += (cols * kBM * OUT_BYTES != chunk);
    bad += (cols > 256) + (cols < 1);
    bad += ((BN / 2) % cols != 0);
    if (CBUF)
        bad += (Cfg::kEpiBufs < 2);                             // C loads run ahead
    bad += (Cfg::kAccBufs < 2);
    return bad;
}

template <int CG, int BN, int OUT_BYTES>
int check_bufs()
{
    return check_one<CG, 0, BN, OUT_BYTES>() + check_one<CG, 2, BN, OUT_BYTES>() +
           (CG == 2 ? check_one<CG, 4, BN, OUT_BYTES>() : 0);
}

}  // namespace

extern "C" int tilecfg_violations()
{
    using namespace tcg;
    int bad = 0;
    bad += check_bufs<1, kBN, 4>() + check_bufs<1, kBN, 2>();
    bad += check_bufs<2, kBN, 4>() + check_bufs<2, kBN, 2>();
    bad += check_bufs<2, kBNNarrow, 4>() + check_bufs<2, kBNNarrow, 2>();
    // the in-kernel TF32 rounding's sub-units: whole 64 x 64 transposes and whole stages
    bad += (kCvK % 64 != 0) + (kCvK % (kDepth * (kRowBytes / 4)) != 0) + (kCvRows != 64);
    return bad;
}

extern "C" int chunk_columns(int out_bytes, int c_bufs)
{
    return tcg::epi_cols(out_bytes, c_bufs);
}
