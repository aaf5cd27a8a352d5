// layout.h -- tile configurations, the shared-memory plan of one CTA, and
// argument validation for the pipelined GEMM.  Pure host/device C++ with no
// CUDA calls, so the same rules are usable without a GPU.
#pragma once

#include <cstdint>

namespace tg {

// Status codes (mirror of tgemm_status_code in the public header).
enum : int {
    kOk = 0,
    kErrInvalidArg = 1,
    kErrUnsupportedDtype = 2,
    kErrAlignment = 3,
    kErrSmemBudget = 4,
    kErrNoKernel = 5,
    kErrArch = 6,
    kErrCuda = 7,
    kErrTimeout = 8,
    kErrCheck = 9,  // an internal bounds or alignment check failed (debug-check builds only)
};

enum : int { kF16 = 0, kBF16 = 1, kF32 = 2 };

constexpr int kThreads = 352;         // 11 warps: TMA producer (A), MMA issuer, 8 epilogue warps,
                                      // TMA producer (B)
constexpr int kProducerBWarp = 10;    // the warp that loads B
constexpr int kEpiWarps = 8;          // two per TMEM lane quarter, splitting the column chunks
constexpr int kEpiCols = 32;          // accumulator columns per epilogue chunk
constexpr int kTmemColsMax = 512;     // tensor-memory columns per SM
constexpr uint32_t kSmemAlign = 1024; // swizzle-atom alignment of every tile slot

inline int dtype_bytes(int dt) { return dt == kF32 ? 4 : (dt == kF16 || dt == kBF16) ? 2 : 0; }

struct Layout {
    int bm, bn, bk, stages;
    int pair;                // 1: two CTAs (a cluster of 2) share one block_M = 256 tile
    int a_rows, b_rows;      // operand rows one CTA holds per slot (pair: 128 and block_N / 2)
    int in_bytes, out_bytes;
    uint32_t a_stage_bytes;  // bm * bk * in_bytes
    uint32_t b_stage_bytes;  // bn * bk * in_bytes
    uint32_t c_buf_bytes;    // one staging buffer: one store box, 32 rows of 64 bytes (32 16-bit or 16 fp32 columns)
    int epi_bufs;            // staging buffers per epilogue warp: 2
    uint32_t off_a, off_b, off_c, off_bar;
    uint32_t bar_bytes;
    uint32_t total;          // bytes requested, including alignment slack
    int64_t bound;           // stages * (A tile + B tile): the budget rule's bound
    int m_halves;            // MMAs along M per k-step: 2 for a one-CTA 256-row tile, else 1
    int quarter_rows;        // accumulator rows per TMEM lane quarter: 32, or 16 for 64-row tiles
    int n_halves;            // pair tiles wider than one MMA (block_N > 256): two MMAs of N = block_N / 2
    int acc_cols;            // TMEM columns of one accumulator (m_halves * bn)
    int acc_stages;          // accumulators in flight (2 lets the epilogue overlap the next tile)
    int tmem_cols;           // power of two >= 32 allocated per CTA
    int swizzle_bytes;       // bytes of one operand row within a K-panel: 32, 64 or 128
    int panels;              // K-panels per slot: 1, or 2 when a row is 256 bytes
};

inline uint32_t round_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Tile shapes the kernel implements: M = 64 or M = 128 MMAs (a 256-row tile
// issues two M = 128 MMAs per k-step), N a multiple of 32 up to the MMA
// maximum of 256, and block_K such that a
// K-contiguous operand row is one swizzle span (32, 64 or 128 bytes) or two
// 128-byte spans (block_K = 128 for 16-bit operands: the slot then holds two
// K-panels of 64 elements, each a standard 128-byte-swizzled tile).  The
// CTA-pair mode implements only block_M = 256 (one M = 256 MMA over the two
// CTAs' 128-row halves), and also tiles of 288 to 512 columns in steps of 32:
// two MMAs of N = block_N / 2 (a multiple of 16) per k-step that share the A
// operand, so each SM pulls up to a quarter less operand data per FLOP than
// with 256 columns.  Each CTA then holds block_N / 4 rows of each N-half of B,
// a whole number of 8-row swizzle atoms.
inline bool tile_supported(int bm, int bn, int bk, int in_bytes, int pair = 0)
{
    if (pair && bm != 256) return false;
    if (bm != 64 && bm != 128 && bm != 256) return false;
    const bool wide = pair && bn > 256 && bn <= 512 && bn % 32 == 0;
    if (!wide && (bn < 32 || bn > 256 || bn % 32 != 0)) return false;
    int row = bk * in_bytes;
    return (row == 32 || row == 64 || row == 128 || row == 256) && bk > 0;
}

// Barrier block: full[S], empty[S], acc_full[2], acc_empty[2], drain, stall,
// epi (the epilogue warps' own barrier), bulk (the in-kernel split
// reduction's copies) (8 bytes each), then the TMEM base address word, the
// abort flag, and a word through which one epilogue thread tells the others
// whether its CTA counted in last (stream-K and in-kernel split reductions),
// plus padding.
inline uint32_t barrier_block_bytes(int stages) { return round_up((2u * stages + 8u) * 8u + 16u, 16u); }

inline Layout make_layout(int bm, int bn, int bk, int stages, int dtype, int out_dtype, int pair = 0)
{
    Layout L{};
    L.bm = bm;
    L.bn = bn;
    L.bk = bk;
    L.stages = stages;
    L.pair = pair ? 1 : 0;
    L.a_rows = pair ? bm / 2 : bm;
    L.b_rows = pair ? bn / 2 : bn;
    L.in_bytes = dtype_bytes(dtype);
    L.out_bytes = dtype_bytes(out_dtype);
    L.a_stage_bytes = uint32_t(L.a_rows) * bk * L.in_bytes;
    L.b_stage_bytes = uint32_t(L.b_rows) * bk * L.in_bytes;
    // The pages' bound for the operand tiles one CTA (one block) holds.
    L.bound = int64_t(stages) * (int64_t(L.a_rows) * bk + int64_t(bk) * L.b_rows) * L.in_bytes;
    L.c_buf_bytes = 32u * 64u;
    L.epi_bufs = 2;
    L.off_a = 0;
    L.off_b = L.off_a + uint32_t(stages) * round_up(L.a_stage_bytes, kSmemAlign);
    L.off_c = L.off_b + uint32_t(stages) * round_up(L.b_stage_bytes, kSmemAlign);
    L.off_bar = L.off_c + round_up(uint32_t(kEpiWarps * L.epi_bufs) * L.c_buf_bytes, kSmemAlign);
    L.bar_bytes = barrier_block_bytes(stages);
    L.total = L.off_bar + L.bar_bytes + kSmemAlign;  // slack to align the dynamic base
    L.m_halves = pair || bm < 256 ? 1 : 2;
    // An M = 64 accumulator keeps its rows in lanes 0-15 of each 32-lane
    // quarter of tensor memory: row r in lane 32 * (r / 16) + r % 16.
    L.quarter_rows = bm == 64 ? 16 : 32;
    L.n_halves = pair && bn > 256 ? 2 : 1;
    L.acc_cols = L.m_halves * bn;
    L.acc_stages = (2 * L.acc_cols <= kTmemColsMax) ? 2 : 1;
    int need = L.acc_stages * L.acc_cols;
    int cols = 32;
    while (cols < need) cols <<= 1;
    L.tmem_cols = cols;
    L.swizzle_bytes = bk * L.in_bytes > 128 ? 128 : bk * L.in_bytes;
    L.panels = bk * L.in_bytes / L.swizzle_bytes;
    return L;
}

// Every check of tgemm_validate, in the documented order.
// Largest number of K splits a plan accepts.
constexpr int kMaxSplits = 64;
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1 - 256;  // largest M, N or K
constexpr int64_t kMaxUnits = int64_t(1) << 30;             // largest tiles x splits

// Effective number of K splits: at least one k-block per split.
inline int effective_splits(int64_t K, int bk, int splits)
{
    const int64_t kb = (K + bk - 1) / bk;
    if (splits <= 1 || kb <= 1) return 1;
    const int64_t per = (kb + splits - 1) / splits;
    return int((kb + per - 1) / per);
}

// In-kernel split-K reduction (kernel mode 2): the K splits of a tile are
// taken by clusters of csk CTAs, which exchange their partial accumulators
// through distributed shared memory.  csk must be 2, 4 or 8 (clusters of up
// to 8 are portable), with one CTA per 128-row tile, a whole number of
// clusters per tile, and slices of block_N / csk columns that are whole
// 32-column epilogue chunks.  Each CTA receives csk parts of 128 x slice
// fp32 values, 128 x block_N x 4 bytes in all, into its operand ring.
inline bool csplit_supported(int bm, int bn, int pair, int eff_splits, int csk)
{
    if (csk != 2 && csk != 4 && csk != 8) return false;
    if (pair || bm != 128) return false;
    if (eff_splits % csk != 0) return false;
    return bn % csk == 0 && (bn / csk) % kEpiCols == 0 && bn / csk <= 128;
}

// B shared by two CTA pairs (kernel mode 3, clusters of 4): the pairs take
// M-adjacent tiles of one N-block, so the CTAs of rank r and r ^ 2 hold the
// same rows of B.  Each loads one part of its B box and multicasts it to both:
// rows [0, part0) from the first pair, [part0, b_box_rows) from the second,
// each part a whole number of 8-row swizzle atoms.
inline int mcast_part0(int b_box_rows) { return (b_box_rows / 2 + 7) / 8 * 8; }
inline bool mcast_supported(int bm, int bn, int pair, int eff_splits, int csk)
{
    if (!pair || bm != 256 || eff_splits != 1 || csk > 1) return false;
    const int box = bn > 256 ? bn / 4 : bn / 2;  // a CTA's rows of one B box (per N-half)
    const int p0 = mcast_part0(box);
    return box % 8 == 0 && p0 >= 8 && box - p0 >= 8;
}

inline int validate(int64_t M, int64_t N, int64_t K, int dtype, int out_dtype, int bm, int bn, int bk,
                    int stages, int64_t smem_limit, int pair = 0, int splits = 1, int csk = 0, int mcast = 0)
{
    if (dtype != kF16 && dtype != kBF16) return kErrUnsupportedDtype;
    if (out_dtype != kF32 && out_dtype != dtype) return kErrUnsupportedDtype;
    // Tile and panel coordinates are 32-bit TMA coordinates: rounded up to a
    // whole tile (at most 256) they must stay below 2^31.
    const int64_t lim = kMaxDim;
    if (M < 0 || N < 0 || K < 0 || M > lim || N > lim || K > lim) return kErrInvalidArg;
    if (stages < 1) return kErrInvalidArg;
    if ((K * dtype_bytes(dtype)) % 16 != 0) return kErrAlignment;
    if ((N * dtype_bytes(out_dtype)) % 16 != 0) return kErrAlignment;
    if (!tile_supported(bm, bn, bk, dtype_bytes(dtype), pair)) return kErrNoKernel;
    if (splits < 1 || splits > kMaxSplits) return kErrInvalidArg;
    // Split s writes its partial tile at workspace row s * ceil(M / bm) * bm + r,
    // also a 32-bit TMA coordinate.
    const int eff = effective_splits(K, bk, splits);
    if (eff > 1 && int64_t(eff) * ((M + bm - 1) / bm) * bm > (int64_t(1) << 31) - 1) return kErrInvalidArg;
    // Work units (tiles x splits) are counted in 32-bit integers by the
    // persistent schedule, with room for one more stride of CTAs.
    if (((M + bm - 1) / bm) * ((N + bn - 1) / bn) * int64_t(eff) > kMaxUnits) return kErrInvalidArg;
    if (stages > 64) return kErrSmemBudget;  // keeps the layout arithmetic in 32 bits
    if (csk > 1 && !csplit_supported(bm, bn, pair, eff, csk)) return kErrInvalidArg;
    // The last M-block pair of an odd tile count has a second tile past M: its
    // rows, up to one more 256-row block, are still 32-bit TMA coordinates.
    if (mcast && (!mcast_supported(bm, bn, pair, eff, csk) || M > kMaxDim - 512)) return kErrInvalidArg;
    // A split-K kernel that reduces through the workspace stages fp32 partial
    // tiles whatever the final output type.
    const int staged = eff > 1 && csk <= 1 ? kF32 : out_dtype;
    Layout L = make_layout(bm, bn, bk, stages, dtype, staged, pair);
    if (L.bound > smem_limit || int64_t(L.total) > smem_limit) return kErrSmemBudget;
    // The cluster exchange lands in the operand ring.
    if (csk > 1 && int64_t(128) * bn * 4 > int64_t(L.off_c - L.off_a)) return kErrSmemBudget;
    return kOk;
}

}  // namespace tg
