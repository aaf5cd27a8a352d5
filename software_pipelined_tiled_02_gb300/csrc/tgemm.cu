// tgemm.cu -- software-pipelined tiled GEMM for GB300 (sm_103a) and its C ABI.
//
// C[M,N] = A[M,K] . B[N,K]^T, fp16/bf16 operands, fp32 accumulation in tensor
// memory, fp32 or 16-bit output.  The computation is the tiled GEMM of the
// TileLang tutorial, chapter 11 "Pipeline and autotuning" (section 1.1: per
// output tile, clear an fp32 accumulator, walk K in block_K steps, copy an A
// tile and a B tile to shared memory, multiply with transpose_B, write the
// tile out).  Its pipelining (sections 2.3, 4.3, 4.4, 5.2) is realised here
// for Blackwell rather than by a compiler pass:
//
//  * the num_stages multi-buffer ("version dimension", slot ko % num_stages)
//    is a ring of num_stages shared-memory slots, each holding one A tile and
//    one B tile in the 32/64/128-byte swizzled K-major layout that both the
//    TMA engine writes and the tensor core reads;
//  * the synchronisation rule of section 5.2 (before writing slot s wait for
//    its last reader; before reading slot s wait for its writer) is a pair of
//    mbarriers per slot: full[s] completes when the TMA bytes of the slot have
//    landed (transaction count), empty[s] completes when the MMAs that read
//    the slot have finished (tcgen05.commit);
//  * the prologue / steady state / epilogue of section 4.3 are implicit: the
//    producer warps run up to num_stages k-blocks ahead of the MMA warp and
//    block only on empty[s];
//  * num_stages = 1 is the unpipelined control of section 1.1 (copy and math
//    serialise on the single slot).
//
// Warp roles (352 threads, one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer of A, which also arms each slot's full barrier
//               (lane 0 runs the loop alone)
//   warp 10     TMA producer of B (lane 0 runs the loop alone)
//   warp 1      TMEM allocator and tcgen05.mma issuer (the converged warp; one
//               elected lane issues)
//   warps 2..9  epilogue, two warps per TMEM lane quarter: TMEM -> registers ->
//               swizzled shared staging -> TMA store
// Each launch is a programmatic dependent of the kernel before it in the
// stream: the set-up overlaps that kernel's end, and every thread waits for
// its writes (griddepcontrol.wait) before any global memory access.
// The accumulator is double-buffered in TMEM when it fits, so the epilogue of
// tile i overlaps the main loop of tile i+1.  The summation order inside a
// tile depends only on the tile shape (k-block by k-block, 16 at a time), never
// on num_stages or the schedule, so results are bit-identical across depths.
//
// Launch shapes (tgemm_kernel<MODE>): one CTA per tile, or CTA pairs
// (cta_group::2, M = 256 over two SMs), or clusters of two pairs that share B
// through TMA multicast, persistent over work units; or one CTA per (tile,
// K split) in thread-block clusters that reduce their splits through
// distributed shared memory.  Split K is otherwise reduced by a
// second kernel or, after a grid-wide barrier, by this one.  The persistent
// schedule can also share the tiles of a partial last wave out by k-blocks
// (a stream-K tail).  Every such combination adds partial sums in an order
// fixed by the shape and the options alone.
//
// Every mbarrier wait is bounded by a %globaltimer watchdog: on expiry the
// kernel records TGEMM_ERR_TIMEOUT in the plan's status word, stops issuing
// work, waits (bounded) for its copies and MMAs in flight, frees its tensor
// memory and returns.  Nothing traps.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <type_traits>

#include "layout.h"
#include "ptx.cuh"
#include "tgemm.h"

namespace tg {

struct Params {  // 64-byte aligned through its CUtensorMap members
    CUtensorMap tmA, tmB, tmC;
    CUtensorMap tmB1;           // mode 3: B's second multicast part (rows part0 .. b_box_rows)
    int M, N, K;
    int num_kb;                 // ceil(K / bk)
    int tiles_m, tiles_n, num_tiles, group_m;
    int splits, kb_per_split;   // K splits per tile (1: none) and k-blocks per split
    int prefetch;               // producer lead in k-blocks, 1..stages (stages: the full ring)
    int split_rows;             // workspace rows per split: tiles_m * block_M, so a tile's
                                // ragged tail stays inside its own split's rows
    int num_units;              // work units: num_tiles * splits
    int bm, bn, bk, stages;
    int n_kstep;                // bk / 16 MMAs along K per slot
    int m_halves;               // MMAs along M per k-step: 2 for a one-CTA 256-row tile, else 1
                                // (pair mode: one M = 256 MMA covers both CTAs)
    int quarter_rows;           // accumulator rows per TMEM lane quarter: 32, or 16 for M = 64
                                // (lanes 0-15 of each quarter hold them)
    int mma_per_kstep;          // MMAs per k-step: 2 M-halves (one CTA, bm = 256), 2 N-halves
                                // (pair, bn > 256), else 1
    uint32_t acc_step;          // TMEM columns between the accumulators of the two MMAs
    uint32_t a_half16, b_half16; // descriptor offsets (16-byte units) of the second MMA's A and B
    int n_halves;               // B boxes per K-panel: 2 for pair tiles wider than 256
    int b_box_rows;             // rows of one B box (b_rows / n_halves)
    int a_rows, b_rows;         // operand rows this CTA loads per slot (pair: 128 and bn / 2)
    int out_mode;               // 0 fp32, 1 fp16, 2 bf16
    int acc_stages, acc_cols, tmem_cols;
    uint32_t idesc;             // tcgen05 instruction descriptor (kind::f16)
    uint32_t a_slot, b_slot;    // bytes between consecutive ring slots
    uint32_t stage_tx;          // bytes the TMA delivers per slot (A box + B box)
    uint32_t row_bytes;         // bytes of one operand row within a K-panel (the swizzle span)
    int panels, panel_k;        // K-panels per slot (1 or 2) and elements per panel
    uint32_t a_panel16, b_panel16;  // distance between a slot's K-panels, in 16-byte units
    uint32_t off_a, off_b, off_c, off_bar, c_buf_bytes;
    int epi_bufs;               // staging buffers per epilogue warp (1 or 2)
    uint32_t desc_lo_flags;     // leading-byte-offset field of the smem descriptor
    uint32_t desc_hi;           // high word: stride byte offset, version, swizzle mode
    unsigned long long watchdog_ns;
    int *status;                // 4 ints: code, role, block, iteration
    int debug_stall;
    // In-kernel split-K reduction (kernel mode 2): the splits of a tile are
    // taken by clusters of csk CTAs, outer = splits / csk clusters per tile.
    int csk, outer;
    int slice_w;                // output columns each CTA of a cluster reduces (block_N / csk)
    float *ws;                  // outer > 1: [outer][split_rows][N] fp32 cluster partials
    int *counters;              // outer > 1: [num_tiles][csk] arrival counts, zero between launches
    void *C;                    // the output, written with plain stores in mode 2
    int stream_ops;             // 1: operand loads carry an L2 evict-first hint
    // K splits reduced inside the kernel after a grid-wide barrier (cooperative
    // launch): grid_bar = {arrivals, generation}, zero between launches.
    int grid_reduce;
    uint32_t *grid_bar;
    int out_mode_final;         // C's type (0 fp32, 1 fp16, 2 bf16); out_mode is what the tiles store
    // Persistent schedule: `workers` CTAs (or pairs) take work units round robin:
    // units 0 .. dp_units-1 whole.  With a stream-K tail, the last sk_tiles
    // tiles' k-blocks are shared out as equal contiguous runs, one per worker.
    int workers, dp_units, sk_tiles;
    int sk_rows;                // rows of a tile one CTA holds (its part of a stream-K partial)
    float *sk_ws;               // [workers][2][ranks][sk_rows][bn] fp32 partial pieces
    int *sk_cnt;                // [sk_tiles][ranks] arrival counts, zero between launches
    // M-blocks of the persistent schedule: tiles_m, or in mode 3 (two CTA pairs
    // per cluster sharing B) ceil(tiles_m / 2) blocks of two M-adjacent tiles.
    int sched_m;
    int b_part0;                // mode 3: rows of B's first multicast part (tmB's box)
};

// ---------------------------------------------------------------- device side

__device__ __forceinline__ void report(const Params &p, int code, int role, int iter)
{
    if (atomicCAS(p.status, 0, code) == 0) {
        p.status[1] = role;
        p.status[2] = int(blockIdx.x);
        p.status[3] = iter;
    }
}

// Debug-check builds (TGEMM_DEBUG_CHECKS=1) test every shared-memory, tensor-
// memory and TMA address the kernel forms against the plan's layout before the
// access.  A failed check records TGEMM_ERR_CHECK with the role and the
// iteration, raises the CTA's abort flag and skips the access, so a bug shows
// up as a status code, never as a fault.  Release builds compile the checks
// away.
#ifndef TGEMM_DEBUG_CHECKS
#define TGEMM_DEBUG_CHECKS 0
#endif

__device__ __forceinline__ bool check(bool ok, const Params &p, volatile int *abort, int role, int iter)
{
    if (TGEMM_DEBUG_CHECKS && !ok) {
        report(p, kErrCheck, role, iter);
        *abort = 1;
        return false;
    }
    return true;
}

// Bounded wait for the phase of parity `parity` of `bar`.  Returns false when
// the CTA has aborted (if honour_abort) or when the watchdog expires; the
// latter is recorded and raises the CTA's abort flag.
__device__ __noinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Params &p, volatile int *abort,
                                      int role, int iter, bool honour_abort = true)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    uint32_t spins = 0;
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((++spins & 15u) == 0) {
            if (honour_abort && *abort) return false;
            if (globaltimer() - t0 > p.watchdog_ns) {
                *abort = 1;
                report(p, kErrTimeout, role, iter);
                return false;
            }
        }
    }
}

// Warp-collective form of wait_bar: every lane polls once (the common case
// is a phase that has already completed); otherwise lane 0 waits with the
// watchdog and the outcome is broadcast, so the warp stays converged and its
// control flow uniform.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Params &p, volatile int *abort,
                                          int role, int iter, bool honour_abort = true)
{
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    int ok = 1;
    if ((threadIdx.x & 31u) == 0) ok = wait_bar(bar, parity, p, abort, role, iter, honour_abort) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ void tile_coords(const Params &p, int t, int &m_blk, int &n_blk)
{
    const int group_tiles = p.group_m * p.tiles_n;
    const int g = t / group_tiles;
    const int first_m = g * p.group_m;
    const int gm = min(p.group_m, p.sched_m - first_m);
    const int r = t - g * group_tiles;
    m_blk = first_m + r % gm;
    n_blk = r / gm;
}

// Work unit u = (tile, K split): its tile, its k-block range [kb0, kb1) and
// the row offset of its output (split s writes rows s*R .. s*R+R-1 of the
// partial-sum workspace, R = tiles_m * block_M >= M; 0 without splitting).
struct Unit {
    int mb, nb, kb0, kb1, row_off;
    int sk;       // 1: a piece of a stream-K tile (k-blocks kb0 .. kb1-1 of it)
    int sk_tile;  // that tile's index among the stream-K tiles
};

__device__ __forceinline__ Unit unit_coords(const Params &p, int u)
{
    Unit w;
    const int tile = u / p.splits;
    const int split = u - tile * p.splits;
    tile_coords(p, tile, w.mb, w.nb);
    w.kb0 = split * p.kb_per_split;
    w.kb1 = min(p.num_kb, w.kb0 + p.kb_per_split);
    w.row_off = split * p.split_rows;
    return w;
}

// Stream-K tail.  The tail's tiles have sk_tiles x num_kb k-block iterations
// in all, tile by tile; worker w takes iterations [I*w/W, I*(w+1)/W), fewer
// than one tile's worth, so at most two tiles.  Tile t's pieces belong to the
// workers sk_lo(t) .. sk_hi(t), in k order.
__device__ __forceinline__ int64_t sk_start(const Params &p, int w)
{
    return int64_t(p.sk_tiles) * p.num_kb * w / p.workers;
}
__device__ __forceinline__ int sk_lo(const Params &p, int t)
{
    const int64_t I = int64_t(p.sk_tiles) * p.num_kb;
    return int((int64_t(p.workers) * (int64_t(t) * p.num_kb + 1) + I - 1) / I) - 1;
}
__device__ __forceinline__ int sk_hi(const Params &p, int t)
{
    const int64_t I = int64_t(p.sk_tiles) * p.num_kb;
    return int((int64_t(p.workers) * (int64_t(t + 1) * p.num_kb) + I - 1) / I) - 1;
}

// Work item i of worker w (a CTA, or a CTA pair): false once w has no more.
// Whole units come first (round robin over the workers), then w's stream-K
// pieces.  Every role of a CTA walks the same items in the same order.
__device__ __forceinline__ bool work_item(const Params &p, int w, int i, Unit &u)
{
    const int n_whole = w < p.dp_units ? (p.dp_units - w + p.workers - 1) / p.workers : 0;
    if (i < n_whole) {
        u = unit_coords(p, w + i * p.workers);
        u.sk = 0;
        u.sk_tile = 0;
        return true;
    }
    if (p.sk_tiles == 0) return false;
    const int64_t s0 = sk_start(p, w), s1 = sk_start(p, w + 1);
    const int t = int(s0 / p.num_kb) + (i - n_whole);
    if (i - n_whole > 1 || int64_t(t) * p.num_kb >= s1) return false;
    const int64_t base = int64_t(t) * p.num_kb;
    u.kb0 = int((s0 > base ? s0 : base) - base);
    u.kb1 = int((s1 < base + p.num_kb ? s1 : base + p.num_kb) - base);
    tile_coords(p, p.dp_units + t, u.mb, u.nb);
    u.row_off = 0;
    u.sk = 1;
    u.sk_tile = t;
    return true;
}

// Shared-memory matrix descriptor of a K-major swizzled operand tile starting
// at shared address `addr` (bits 0-13: address >> 4; 16-29: leading byte
// offset >> 4; 32-45: stride byte offset >> 4; 46: version 1; 61-63: swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, const Params &p)
{
    const uint32_t lo = ((addr >> 4) & 0x3FFFu) | p.desc_lo_flags;
    return (uint64_t(p.desc_hi) << 32) | lo;
}

struct MmaCtx {
    uint32_t sA, sB, tmem, bars;
    int S;
    uint32_t stall, drain;
    int unit0, ustride;  // first tile and tile stride of this CTA (or CTA pair)
    // pair mode: CTAs whose barriers a commit arrives on -- every CTA that
    // loads into this pair's slots (empty), the pair (acc_full), this CTA (drain)
    uint16_t empty_mask, pair_mask, self_mask;
};

// The MMA warp's main loop.  NK = MMAs of K = 16 per ring slot (block_K / 16),
// MH = MMAs per k-step: the two M = 128 halves of a one-CTA 256-row tile (the
// second reads A 128 rows further on and writes the accumulator block_N
// columns further on), or in pair mode the two N-halves of a tile wider than
// 256 columns (the second reads the second half of this CTA's B rows and
// writes block_N / 2 columns further on); 1 otherwise.  Descriptors of slot s
// are the slot-0 descriptors plus s slot strides (address field in 16-byte
// units); k-step kk adds 32 bytes.  In pair mode this runs in the even CTA
// only: its commits arrive on the barriers of both CTAs.  The whole warp runs
// the loop converged, and elect.sync inside each MMA and commit picks the lane
// that issues it.  With lane 0 alone issuing under a branch, the issue path
// took about 360 cycles per slot plus 69 per MMA (clock64 probe), more than the
// tensor core's time for slots of under ~900 MMA cycles: 448 for a 256x224x64
// pair tile, 704 for 256x352x64.  Elected issue takes about 35 per MMA.
template <int NK, int MH, bool PAIR>
__device__ __forceinline__ void mma_role(const Params &p, const MmaCtx &c, volatile int *abort, int lane)
{
    const int S = c.S;
    auto full = [&](int s) { return c.bars + 8u * uint32_t(s); };
    auto empty = [&](int s) { return c.bars + 8u * uint32_t(S + s); };
    auto acc_full = [&](int a) { return c.bars + 8u * uint32_t(2 * S + a); };
    auto acc_empty = [&](int a) { return c.bars + 8u * uint32_t(2 * S + 2 + a); };
    auto mma = [&](uint32_t d, uint64_t ad, uint64_t bd, uint32_t acc) {
        if constexpr (PAIR)
            mma_f16_pair(d, ad, bd, p.idesc, acc);
        else
            mma_f16(d, ad, bd, p.idesc, acc);
    };
    auto commit_both = [&](uint32_t bar, uint16_t mask) {
        if constexpr (PAIR)
            mma_commit_pair_elect(bar, mask);
        else
            mma_commit_elect(bar);
    };
    const uint64_t ad0 = smem_desc(c.sA, p), bd0 = smem_desc(c.sB, p);
    const uint64_t a_step = p.a_slot >> 4, b_step = p.b_slot >> 4;
    const uint64_t a_half = p.a_half16, b_half = p.b_half16;
    const uint64_t a_panel = p.a_panel16, b_panel = p.b_panel16;
    int s = 0;
    uint32_t ph = 0;
    uint64_t ad = ad0, bd = bd0;
    int a = 0;
    uint32_t aph = 0;
    int it = 0;
    bool ok = true;
    if (p.debug_stall) ok = warp_wait(c.stall, 0, p, abort, 1, 0);  // test hook: nothing arrives
    for (int i = 0; ok; ++i) {
        Unit w;
        if (!work_item(p, c.unit0, i, w)) break;
        const int kb0 = w.kb0, kb1 = w.kb1;
        if (!warp_wait(acc_empty(a), aph ^ 1u, p, abort, 1, it)) break;
        tc_fence_after();
        const uint32_t d = c.tmem + uint32_t(a * p.acc_cols);
        const uint32_t d2 = d + p.acc_step;
        for (int kb = kb0; kb < kb1; ++kb) {
            if (!warp_wait(full(s), ph, p, abort, 1, it)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // slot s's operands lie inside the A and B rings; the accumulator inside TMEM.
            // The descriptor holds address bits 4-17 of this CTA's shared window; in a
            // cluster the window's addresses also carry the CTA's rank above them.
            const bool in_range =
                check(uint32_t(ad & 0x3FFFu) << 4 >= (c.sA & 0x3FFFFu) &&
                          ((uint32_t(ad & 0x3FFFu) << 4) + p.a_slot) <= (c.sA & 0x3FFFFu) + uint32_t(S) * p.a_slot &&
                          uint32_t(bd & 0x3FFFu) << 4 >= (c.sB & 0x3FFFFu) &&
                          ((uint32_t(bd & 0x3FFFu) << 4) + p.b_slot) <= (c.sB & 0x3FFFFu) + uint32_t(S) * p.b_slot &&
                          (a + 1) * p.acc_cols <= p.tmem_cols && kb1 <= p.num_kb,
                      p, abort, 1, it);
            if (in_range) {
                const uint32_t first = kb != kb0 ? 1u : 0u;
#pragma unroll
                for (int kk = 0; kk < NK; ++kk) {
                    // k-step kk: 32-byte step (kk % 4) inside K-panel kk / 4
                    const uint64_t ka = uint64_t(2 * (kk & 3)) + uint64_t(kk >> 2) * a_panel;
                    const uint64_t kb_ = uint64_t(2 * (kk & 3)) + uint64_t(kk >> 2) * b_panel;
#pragma unroll
                    for (int h = 0; h < MH; ++h)
                        mma(h ? d2 : d, ad + ka + (h ? a_half : 0), bd + kb_ + (h ? b_half : 0), kk == 0 ? first : 1u);
                }
                commit_both(empty(s), c.empty_mask);  // slot s may be refilled once these MMAs finish
            }
            __syncwarp();
            ++it;
            if (++s == S) {
                s = 0;
                ph ^= 1u;
                ad = ad0;
                bd = bd0;
            } else {
                ad += a_step;
                bd += b_step;
            }
        }
        if (!ok) break;
        commit_both(acc_full(a), c.pair_mask);  // accumulator a is complete (in both CTAs)
        __syncwarp();
        if (++a == p.acc_stages) {
            a = 0;
            aph ^= 1u;
        }
    }
    // Every MMA this warp issued must finish before TMEM is freed.
    if (lane == 0) {
        if constexpr (PAIR)
            mma_commit_pair(c.drain, c.self_mask);
        else
            mma_commit(c.drain);
        wait_bar(c.drain, 0, p, abort, 1, it, false);
    }
    __syncwarp();
}

template <int MH, bool PAIR>
__device__ __forceinline__ void mma_dispatch_nk(const Params &p, const MmaCtx &c, volatile int *abort, int lane)
{
    switch (p.n_kstep) {
    case 1: mma_role<1, MH, PAIR>(p, c, abort, lane); break;
    case 2: mma_role<2, MH, PAIR>(p, c, abort, lane); break;
    case 4: mma_role<4, MH, PAIR>(p, c, abort, lane); break;
    default: mma_role<8, MH, PAIR>(p, c, abort, lane); break;
    }
}

// K-split reduction inside the kernel (modes 0 and 1, grid_reduce).  The
// launch is cooperative, so every CTA of the grid is resident at once and a
// grid-wide barrier cannot wait forever for a CTA that has not started.
// After its last unit, each CTA's epilogue has stored its fp32 partial tiles
// to the workspace; thread 0 of the epilogue counts the CTA in, and the last
// arrival opens the barrier by advancing its generation.  Then the epilogue
// threads of all CTAs split the M x N outputs among themselves and add, for
// each, its partials in split order 0, 1, ..., splits-1 -- the order of the
// separate reduction kernel, so both give the same bits -- and round once to
// C's type.  The barrier resets itself (arrivals back to 0), so launches need
// no host-side state; its wait is bounded by the watchdog.
__device__ __noinline__ void grid_reduce_phase(const Params &p, volatile int *abort, int *flag, uint32_t sA,
                                               uint32_t bulk_bar)
{
    const int et = int(threadIdx.x) - 2 * 32;  // 0..255 over the eight epilogue warps
    if ((threadIdx.x & 31u) == 0) {
        fence_proxy_async_global();  // this warp's completed partial stores, before the count below
        __threadfence();
    }
    named_bar_sync(1, 8 * 32);
    if (et == 0) {
        uint32_t *count = p.grid_bar, *gen = p.grid_bar + 1;
        const uint32_t g0 = ld_acquire_gpu(gen);
        __threadfence();
        if (atomicAdd(count, 1u) == gridDim.x - 1) {
            *count = 0u;                 // the next launch starts from no arrivals
            __threadfence();
            st_release_gpu(gen, g0 + 1u);  // open the barrier
        } else {
            const uint64_t t0 = globaltimer();
            uint32_t spins = 0;
            while (ld_acquire_gpu(gen) == g0) {
                if ((++spins & 63u) == 0 && globaltimer() - t0 > p.watchdog_ns) {
                    report(p, kErrTimeout, 2, -1);
                    *abort = 1;
                    break;
                }
            }
        }
        *flag = *abort ? 0 : 1;
    }
    named_bar_sync(1, 8 * 32);
    if (!*reinterpret_cast<volatile int *>(flag)) return;
    __threadfence();
    // CTA b reduces a contiguous run of the M x N outputs, in 16-byte groups:
    // [b * per, (b + 1) * per).  Split s's partial of output e sits at
    // ws[s * split_rows * N + e].  One thread copies the run of every split
    // into this CTA's operand ring (idle now: all its MMAs are done) with
    // bulk copies on one mbarrier; then the epilogue threads add the splits
    // in order 0, 1, ..., splits-1 from shared memory and round once to C's
    // type.  Runs longer than the ring allows are done in rounds.
    const int64_t n4 = int64_t(p.M) * p.N / 4;
    const int64_t per = (n4 + gridDim.x - 1) / gridDim.x;
    const int64_t b0 = int64_t(blockIdx.x) * per;
    const int64_t b1 = b0 + per < n4 ? b0 + per : n4;
    const int64_t stride4 = int64_t(p.split_rows) * p.N / 4;
    const float4 *W = reinterpret_cast<const float4 *>(p.ws);
    const int64_t chunk = int64_t(p.off_c - p.off_a) / 16 / p.splits;  // 16-byte groups per split per round
    uint32_t ph = 0;
    for (int64_t c0 = b0; c0 < b1; c0 += chunk) {
        const int64_t cnt = b1 - c0 < chunk ? b1 - c0 : chunk;
        named_bar_sync(1, 8 * 32);  // the previous round's reads of the ring are done
        if (et == 0) {
            fence_proxy_async_global();  // the partials, read through the async proxy below
            mbar_arrive_expect_tx(bulk_bar, uint32_t(cnt * 16 * p.splits));
            for (int s = 0; s < p.splits; ++s)
                bulk_load(sA + uint32_t(s * chunk * 16), W + int64_t(s) * stride4 + c0, uint32_t(cnt * 16), bulk_bar);
        }
        // Every epilogue warp waits for the copies (bounded: on expiry the wait
        // records the timeout and raises the abort flag), then all meet, so that
        // they read the flag alike and leave together.
        warp_wait(bulk_bar, ph, p, abort, 2, -2, false);
        ph ^= 1u;
        named_bar_sync(1, 8 * 32);
        if (*abort) return;
        for (int64_t i = et; i < cnt; i += 8 * 32) {
            float4 acc = ld_shared_v4f(sA + uint32_t(i * 16));
            for (int s = 1; s < p.splits; ++s) {
                const float4 t = ld_shared_v4f(sA + uint32_t((s * chunk + i) * 16));
                acc.x += t.x;
                acc.y += t.y;
                acc.z += t.z;
                acc.w += t.w;
            }
            const int64_t e = c0 + i;
            if (p.out_mode_final == 0) {
                reinterpret_cast<float4 *>(p.C)[e] = acc;
            } else if (p.out_mode_final == 1) {
                __half2 lo = __floats2half2_rn(acc.x, acc.y), hi = __floats2half2_rn(acc.z, acc.w);
                uint2 u;
                u.x = *reinterpret_cast<uint32_t *>(&lo);
                u.y = *reinterpret_cast<uint32_t *>(&hi);
                reinterpret_cast<uint2 *>(p.C)[e] = u;
            } else {
                __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
                uint2 u;
                u.x = *reinterpret_cast<uint32_t *>(&lo);
                u.y = *reinterpret_cast<uint32_t *>(&hi);
                reinterpret_cast<uint2 *>(p.C)[e] = u;
            }
        }
    }
}

// Epilogue of kernel mode 2 (split K reduced inside the kernel).  This CTA
// holds, in tensor memory, the fp32 partial sum of one K range of its tile
// (128 rows x block_N columns); its cluster holds the csk consecutive K
// ranges o*csk .. o*csk + csk-1 of the same tile, cluster rank r taking
// range o*csk + r.
//  1. Once its own MMAs are done, a cluster barrier: every CTA of the cluster
//     has finished its K loop, so every operand ring in the cluster is idle.
//  2. Reduce-scatter.  CTA r owns the tile's columns [r*slice_w, (r+1)*slice_w).
//     Each CTA copies every 32-column chunk of its accumulator into the ring
//     of the chunk's owner, into the region of its own rank
//     (st.shared::cluster); a second cluster barrier makes the copies visible.
//  3. The owner adds the csk parts of its slice in rank order 0, 1, ..., csk-1.
//  4. outer = 1: it converts and stores the slice to C.  outer > 1: it stores
//     the fp32 slice to the workspace region of its outer index o and counts
//     in on the slice's counter; the CTA that counts last adds the outer
//     partials in order o = 0, 1, ..., outer-1 (its own from shared memory,
//     the others from the workspace), converts, stores to C and resets the
//     counter.  No CTA waits for another outside its own cluster.
// The order of every sum depends on the tile shape, csk and outer only: never
// on num_stages, the schedule or which CTA arrives last.  Every path through
// this function meets both cluster barriers, aborted or not.
//
// A part (one rank's 128 x slice_w values of a slice) is stored column group
// by column group: the 16 bytes of row r, columns 4j .. 4j+3 sit at
// (j * 128 + (r ^ (j % 8))) * 16.  A warp's copy of one column group (its 32
// rows) is then 512 contiguous bytes of the owner's memory, and the owner's
// threads, which take consecutive column groups of one row (so that their
// global stores are contiguous), read eight different bank groups.

// Items (16-byte column groups of one slice row) per epilogue thread:
// 128 x slice_w / 4 over 256 threads = slice_w / 8 -- 4, 8, 12 or 16 for the
// slices of 32, 64, 96 and 128 columns that block_N <= 256 and csk >= 2
// allow; a slice row has 2 x NIT column groups.
template <int NIT>
__device__ __forceinline__ void csplit_finish(const Params &p, uint32_t sA, int *flag, int tile, int o,
                                              uint32_t crank, int grow0, int gcol0, uint32_t part_bytes)
{
    constexpr int CPR = 2 * NIT;                 // column groups per slice row
    const int et = int(threadIdx.x) - 2 * 32;  // 0..255 over the eight epilogue warps
    // Item i of this thread: g = et + 256 i, slice row g / CPR, column group g % CPR.
    auto row_of = [&](int i) { return (et + i * 8 * 32) / CPR; };
    auto grp_of = [&](int i) { return (et + i * 8 * 32) % CPR; };
    auto inside = [&](int i) { return grow0 + row_of(i) < p.M && gcol0 + 4 * grp_of(i) < p.N; };
    auto elem = [&](int i) { return int64_t(grow0 + row_of(i)) * p.N + gcol0 + 4 * grp_of(i); };
    // The cluster's sum of item i, parts added in rank order.
    auto cluster_sum = [&](int i) -> float4 {
        const int r = row_of(i), j = grp_of(i);
        const uint32_t off = (uint32_t(j) * 128u + uint32_t(r ^ (j & 7))) << 4;
        float4 acc = ld_shared_v4f(sA + off);
        for (int src = 1; src < p.csk; ++src) {
            const float4 t = ld_shared_v4f(sA + uint32_t(src) * part_bytes + off);
            acc.x += t.x;
            acc.y += t.y;
            acc.z += t.z;
            acc.w += t.w;
        }
        return acc;
    };
    const int64_t plane = int64_t(p.split_rows) * p.N;  // floats per outer region of the workspace
    float4 tot[NIT];
    if (p.outer > 1) {
        float *wo = p.ws + int64_t(o) * plane;
#pragma unroll
        for (int i = 0; i < NIT; ++i)
            if (inside(i)) *reinterpret_cast<float4 *>(wo + elem(i)) = cluster_sum(i);
        __threadfence();  // this thread's partials are visible GPU-wide before the count below
        named_bar_sync(1, 8 * 32);
        if (et == 0) {
            int *cnt = p.counters + tile * p.csk + int(crank);
            const int last = atomicAdd(cnt, 1) == p.outer - 1;
            if (last) *cnt = 0;  // every cluster of this launch has counted in: ready for the next launch
            *flag = last;
        }
        named_bar_sync(1, 8 * 32);
        if (!*reinterpret_cast<volatile int *>(flag)) return;
        __threadfence();
        // The total in the order o = 0, 1, ..., outer-1; for each outer index
        // all of this thread's loads are issued before any is added.
        for (int oo = 0; oo < p.outer; ++oo) {
            float4 t[NIT];
            if (oo == o) {
#pragma unroll
                for (int i = 0; i < NIT; ++i) t[i] = cluster_sum(i);
            } else {
                const float *wq = p.ws + int64_t(oo) * plane;
#pragma unroll
                for (int i = 0; i < NIT; ++i)  // items outside C read element 0 of the region, never stored
                    t[i] = __ldcg(reinterpret_cast<const float4 *>(wq + (inside(i) ? elem(i) : 0)));
            }
#pragma unroll
            for (int i = 0; i < NIT; ++i) {
                if (oo == 0) {
                    tot[i] = t[i];
                } else {
                    tot[i].x += t[i].x;
                    tot[i].y += t[i].y;
                    tot[i].z += t[i].z;
                    tot[i].w += t[i].w;
                }
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < NIT; ++i) tot[i] = cluster_sum(i);
    }
#pragma unroll
    for (int i = 0; i < NIT; ++i) {
        if (!inside(i)) continue;
        const int64_t e = elem(i);
        const float4 acc = tot[i];
        if (p.out_mode == 0) {
            *reinterpret_cast<float4 *>(static_cast<float *>(p.C) + e) = acc;
        } else if (p.out_mode == 1) {
            __half2 lo = __floats2half2_rn(acc.x, acc.y), hi = __floats2half2_rn(acc.z, acc.w);
            uint2 u;
            u.x = *reinterpret_cast<uint32_t *>(&lo);
            u.y = *reinterpret_cast<uint32_t *>(&hi);
            *reinterpret_cast<uint2 *>(static_cast<__half *>(p.C) + e) = u;
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 u;
            u.x = *reinterpret_cast<uint32_t *>(&lo);
            u.y = *reinterpret_cast<uint32_t *>(&hi);
            *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.C) + e) = u;
        }
    }
}

__device__ __noinline__ void csplit_epilogue(const Params &p, uint32_t sA, int *flag, uint32_t tmem,
                                             uint32_t acc_full0, volatile int *abort, int warp, int lane,
                                             int unit)
{
    const int q = warp & 3;             // TMEM lane quarter: rows 32q .. 32q+31
    const int sub = (warp - 2) >> 2;    // the two warps of a quarter take alternate chunks
    const uint32_t crank = cluster_ctarank();
    const int tile = unit / p.splits;
    const int o = (unit - tile * p.splits) / p.csk;
    const Unit w = unit_coords(p, unit);
    const bool ok = unit < p.num_units && warp_wait(acc_full0, 0, p, abort, 2, 0);
    tc_fence_after();
    __syncwarp();
    cluster_sync();  // 1: every ring of the cluster is idle
    const uint32_t part_bytes = 128u * uint32_t(p.slice_w) * 4u;  // one rank's part of a slice
    if (ok && !*abort) {
        const int row = q * 32 + lane;
        int idx = 0;
        for (int c = 0; c * kEpiCols < p.bn; ++c) {
            if ((idx++ & 1) != sub) continue;
            const int owner = c * kEpiCols / p.slice_w;
            const int j0 = (c * kEpiCols - owner * p.slice_w) / 4;  // first column group of the chunk in the slice
            // the part lies inside the ring (the plan checks csk x part_bytes <= ring bytes)
            if (!check(uint32_t(p.csk) * part_bytes <= p.off_c - p.off_a && owner < p.csk &&
                           uint32_t(j0 + 8) * 128u * 16u <= part_bytes,
                       p, abort, 2, c))
                continue;
            uint32_t v[32];
            if (p.num_kb > 0) {
                tmem_ld_32x32b_x32(tmem + (uint32_t(q * 32) << 16) + uint32_t(c * kEpiCols), v);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0u;
            }
            const uint32_t dst = map_to_rank(sA + crank * part_bytes, uint32_t(owner));
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const uint32_t j = uint32_t(j0 + jj);
                st_cluster_v4(dst + ((j * 128u + uint32_t(row ^ int(j & 7u))) << 4), v[4 * jj], v[4 * jj + 1],
                              v[4 * jj + 2], v[4 * jj + 3]);
            }
        }
    }
    __syncwarp();
    cluster_sync();  // 2: every part is in its owner's ring
    if (!ok || *abort) return;
    const int grow0 = w.mb * p.bm;
    const int gcol0 = w.nb * p.bn + int(crank) * p.slice_w;
    switch (p.slice_w) {
    case 32: csplit_finish<4>(p, sA, flag, tile, o, crank, grow0, gcol0, part_bytes); break;
    case 64: csplit_finish<8>(p, sA, flag, tile, o, crank, grow0, gcol0, part_bytes); break;
    case 96: csplit_finish<12>(p, sA, flag, tile, o, crank, grow0, gcol0, part_bytes); break;
    case 128: csplit_finish<16>(p, sA, flag, tile, o, crank, grow0, gcol0, part_bytes); break;
    default: check(false, p, abort, 2, p.slice_w); break;  // the plan admits no other slice width
    }
}

// One kernel, four launch shapes.
//  MODE 0: one CTA per tile, persistent over work units.
//  MODE 1: clusters of two CTAs; the pair computes one block_M = 256 tile
//    with one M = 256 MMA per k-step issued by the even CTA, each CTA holding
//    128 rows of A, half of B's block_N rows and 128 rows of the accumulator.
//    The pair shares one pipeline: both CTAs' TMA loads complete the even
//    CTA's full[s], and the even CTA's commits arrive on both CTAs' empty[s]
//    and acc_full[a]; both CTAs' epilogues arrive on the even CTA's
//    acc_empty[a].
//  MODE 2: split K reduced inside the kernel.  One CTA per work unit (tile,
//    K split), no persistence; the csk consecutive splits of a tile form one
//    cluster, which sums its partial accumulators through distributed shared
//    memory (csplit_epilogue); clusters of the same tile then combine through
//    global memory, the last to arrive adding all in a fixed order.
//  MODE 3: clusters of four, two CTA pairs as in mode 1 (ranks 0-1 and 2-3)
//    that take the two M-adjacent tiles of one N-block.  The CTAs of rank r
//    and r ^ 2 hold the same B rows; each loads one part of them and TMA
//    multicast writes it into both, completing each receiving pair's even-CTA
//    full[s].  empty[s] counts both pairs' commits, since a slot holds data of
//    both; accumulator hand-offs stay within a pair.
template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) tgemm_kernel(const __grid_constant__ Params p)
{
    constexpr bool PAIR = MODE == 1 || MODE == 3;
    constexpr bool CSPLIT = MODE == 2;
    constexpr bool MC = MODE == 3;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = (kSmemAlign - (raw & (kSmemAlign - 1))) & (kSmemAlign - 1);
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;
    const uint32_t sA = sbase + p.off_a;
    const uint32_t sB = sbase + p.off_b;
    const uint32_t sC = sbase + p.off_c;
    const int S = p.stages;
    const uint32_t bars = sbase + p.off_bar;
    auto full = [&](int s) { return bars + 8u * uint32_t(s); };
    auto empty = [&](int s) { return bars + 8u * uint32_t(S + s); };
    auto acc_full = [&](int a) { return bars + 8u * uint32_t(2 * S + a); };
    auto acc_empty = [&](int a) { return bars + 8u * uint32_t(2 * S + 2 + a); };
    const uint32_t drain = bars + 8u * uint32_t(2 * S + 4);
    const uint32_t stall = bars + 8u * uint32_t(2 * S + 5);
    const uint32_t epi_bar = bars + 8u * uint32_t(2 * S + 6);   // the eight epilogue warps meet here
    const uint32_t bulk_bar = bars + 8u * uint32_t(2 * S + 7);  // the in-kernel split reduction's copies
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + p.off_bar + 8u * uint32_t(2 * S + 8));
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *flag = reinterpret_cast<int *>(tmem_slot + 2);  // "counted in last", for the epilogue warps

    const int warp = int(threadIdx.x) / 32;
    const int lane = int(threadIdx.x) % 32;
    const uint32_t crank = PAIR ? cluster_ctarank() : 0u;  // rank in the cluster
    const uint32_t rank = MC ? crank & 1u : crank;         // in the pair; 0: the MMA-issuing CTA
    const uint32_t leader = MC ? crank & ~1u : 0u;         // the pair's even CTA
    const int pidx = MC ? int(crank >> 1) : 0;             // mode 3: the cluster's first or second pair
    const int unit0 = MC ? int(blockIdx.x >> 2) : PAIR ? int(blockIdx.x >> 1) : int(blockIdx.x);
    const int ustride = MC ? int(gridDim.x >> 2) : PAIR ? int(gridDim.x >> 1) : int(gridDim.x);
    // A work item's tile: in mode 3 the cluster's item is a pair of M-adjacent
    // tiles, the second pair taking the lower one (past M when tiles_m is odd:
    // its A loads read zeros and its rows are not stored).
    auto item = [&](int i, Unit &u) -> bool {
        if (!work_item(p, unit0, i, u)) return false;
        if constexpr (MC) u.mb = 2 * u.mb + pidx;
        return true;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), MC ? 2 : 1);  // mode 3: both pairs release a slot before it refills
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full(a), 1);
            mbar_init(acc_empty(a), PAIR ? 2 * kEpiWarps : kEpiWarps);
        }
        mbar_init(drain, 1);
        mbar_init(stall, 1);
        mbar_init(epi_bar, kEpiWarps);
        mbar_init(bulk_bar, 1);
        *abort = 0;
        fence_mbar_init();
        if (p.num_kb > 0) {
            prefetch_tmap(&p.tmA);
            prefetch_tmap(&p.tmB);
        }
        prefetch_tmap(&p.tmC);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_addr(tmem_slot), uint32_t(p.tmem_cols));
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_addr(tmem_slot), uint32_t(p.tmem_cols));
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // both CTAs' barriers exist before either signals the other
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched as a programmatic dependent of the kernel before it, this one may
    // have started while that kernel finished: nothing above touched global
    // memory, and nothing below may before that kernel's writes are visible.
    griddep_wait();
    // A split-K reduction (or another GEMM) launched after this kernel may be
    // scheduled from now on; it waits for this grid's completion in turn.
    griddep_launch_dependents();

    if (warp == 0 || warp == kProducerBWarp) {
        // ---------------- producers: fill the ring, up to num_stages slots ahead.
        // Warp 0 arms each slot and loads A, warp 10 loads B: a pair-mode
        // (cta_group::2) TMA load takes about 120 cycles to issue, so one
        // thread issuing both operands refilled a block_K = 64 slot more
        // slowly than the MMAs drained it.
        // Pair mode: each CTA loads its own rows of A and B into its own slot;
        // both complete the even CTA's full[s], which the even CTA arms with
        // the bytes of both.
        const uint32_t full_leader = PAIR ? map_to_rank(full(0), leader) : 0u;
        // Streamed operands: each line is read by the tiles that share it at
        // about the same time and not again, so it goes first when L2 needs room.
        const uint64_t policy = p.stream_ops ? policy_evict_first() : 0ull;
        int s = 0;
        uint32_t ph = 0;
        int issued = 0;
        bool ok = true;
        // Prefetch distance D < S: before loading k-block i, also wait until
        // the MMAs of k-block i - D have released their slot (slot (i-D) % S,
        // whose latest use is i - D because (i - D) + S > i).
        const int D = p.prefetch;
        int sd = S - D;  // slot of iteration issued - D, once issued >= D
        uint32_t phd = 0;
        // The whole ring (D = S), the default: lane 0 of each producer warp
        // alone runs a loop whose operand, tile shape (K-panels per slot, B
        // boxes per panel) and load hint are compile-time, with the launch
        // constants in registers.  The loop is a chain of dependent
        // single-thread steps, and each parameter read or branch in it
        // lengthens the time to refill a slot.  Both warps wait for the same
        // empty[s]; B bytes that land before warp 0 arms the phase only take
        // its transaction count below zero until the arming arrives.
        auto lean = [&](auto panels_c, auto nh_c, auto stream_c, auto part_c) {
            constexpr int PANELS = decltype(panels_c)::value;
            [[maybe_unused]] constexpr int NH = decltype(nh_c)::value;
            constexpr bool STREAM = decltype(stream_c)::value;
            constexpr bool LOAD_A = decltype(part_c)::value == 0;  // else B
            const uint32_t a_slot = p.a_slot, b_slot = p.b_slot, tx = p.stage_tx;
            const uint32_t a_pan = p.a_panel16 << 4, b_pan = p.b_panel16 << 4;
            [[maybe_unused]] const uint32_t b_half = p.b_half16 << 4;  // a wide tile's second N-half
            const int bk = p.bk, panel_k = p.panel_k;
            [[maybe_unused]] const int bnh = p.bn >> 1;
            const uint32_t part = MC && pidx ? uint32_t(p.b_part0) * p.row_bytes : 0u;
            const int yp = MC && pidx ? p.b_part0 : 0;
            [[maybe_unused]] const void *bmap = MC && pidx ? &p.tmB1 : &p.tmB;
            [[maybe_unused]] const uint16_t mask = uint16_t((1u << crank) | (1u << (crank ^ 2u)));
            for (int i = 0;; ++i) {
                Unit w;
                if (!item(i, w)) break;
                const int m0 = w.mb * p.bm + int(rank) * p.a_rows;
                const int n0 = w.nb * p.bn + int(rank) * p.b_box_rows + yp;
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (!mbar_try_wait(empty(s), ph ^ 1u) && !wait_bar(empty(s), ph ^ 1u, p, abort, 0, issued)) {
                        ok = false;
                        return;
                    }
                    if (!check(s < S && (kb * bk * 2) % 16 == 0 && kb < p.num_kb &&
                                   w.mb < (MC ? 2 * p.sched_m : p.tiles_m) && w.nb < p.tiles_n &&
                                   PANELS * int(a_pan) <= int(a_slot) && PANELS * int(b_pan) <= int(b_slot),
                               p, abort, 0, issued)) {
                        ok = false;
                        return;
                    }
                    const uint32_t a_dst = sA + uint32_t(s) * a_slot, b_dst = sB + uint32_t(s) * b_slot + part;
                    const uint32_t bar = PAIR ? full_leader + 8u * uint32_t(s) : full(s);
                    if (LOAD_A && (!PAIR || rank == 0)) mbar_arrive_expect_tx(full(s), tx);
#pragma unroll
                    for (int pl = 0; pl < PANELS; ++pl) {
                        const int x = kb * bk + pl * panel_k;
                        const uint32_t a_at = a_dst + uint32_t(pl) * a_pan, b_at = b_dst + uint32_t(pl) * b_pan;
                        if constexpr (LOAD_A) {
                            if constexpr (PAIR) {
                                if constexpr (STREAM)
                                    tma_load_2d_pair_hint(a_at, &p.tmA, x, m0, bar, policy);
                                else
                                    tma_load_2d_pair(a_at, &p.tmA, x, m0, bar);
                            } else if constexpr (STREAM) {
                                tma_load_2d_hint(a_at, &p.tmA, x, m0, bar, policy);
                            } else {
                                tma_load_2d(a_at, &p.tmA, x, m0, bar);
                            }
                        } else if constexpr (PAIR) {
                            if constexpr (MC) {
                                // B: this CTA's part of its rows, multicast to it and to the CTA
                                // of the other pair that holds the same rows (rank ^ 2)
                                if constexpr (STREAM) {
                                    tma_load_2d_pair_mc_hint(b_at, bmap, x, n0, bar, mask, policy);
                                    if constexpr (NH == 2)
                                        tma_load_2d_pair_mc_hint(b_at + b_half, bmap, x, n0 + bnh, bar, mask, policy);
                                } else {
                                    tma_load_2d_pair_mc(b_at, bmap, x, n0, bar, mask);
                                    if constexpr (NH == 2) tma_load_2d_pair_mc(b_at + b_half, bmap, x, n0 + bnh, bar, mask);
                                }
                            } else if constexpr (STREAM) {
                                tma_load_2d_pair_hint(b_at, &p.tmB, x, n0, bar, policy);
                                // a wide tile's second N-half: this CTA's rows of it, block_N / 2 further on
                                if constexpr (NH == 2) tma_load_2d_pair_hint(b_at + b_half, &p.tmB, x, n0 + bnh, bar, policy);
                            } else {
                                tma_load_2d_pair(b_at, &p.tmB, x, n0, bar);
                                if constexpr (NH == 2) tma_load_2d_pair(b_at + b_half, &p.tmB, x, n0 + bnh, bar);
                            }
                        } else if constexpr (STREAM) {
                            tma_load_2d_hint(b_at, &p.tmB, x, n0, bar, policy);
                        } else {
                            tma_load_2d(b_at, &p.tmB, x, n0, bar);
                        }
                    }
                    ++issued;
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        };
        using One = std::integral_constant<int, 1>;
        using Two = std::integral_constant<int, 2>;
        using Plain = std::false_type;
        using Stream = std::true_type;
        using PartA = std::integral_constant<int, 0>;
        using PartB = std::integral_constant<int, 1>;
        if (D >= S && lane == 0) {
            if (warp == 0) {
                if (p.panels == 2)
                    p.stream_ops ? lean(Two{}, One{}, Stream{}, PartA{}) : lean(Two{}, One{}, Plain{}, PartA{});
                else
                    p.stream_ops ? lean(One{}, One{}, Stream{}, PartA{}) : lean(One{}, One{}, Plain{}, PartA{});
            } else if (p.panels == 2) {
                if (p.n_halves == 2)
                    p.stream_ops ? lean(Two{}, Two{}, Stream{}, PartB{}) : lean(Two{}, Two{}, Plain{}, PartB{});
                else
                    p.stream_ops ? lean(Two{}, One{}, Stream{}, PartB{}) : lean(Two{}, One{}, Plain{}, PartB{});
            } else if (p.n_halves == 2) {
                p.stream_ops ? lean(One{}, Two{}, Stream{}, PartB{}) : lean(One{}, Two{}, Plain{}, PartB{});
            } else {
                p.stream_ops ? lean(One{}, One{}, Stream{}, PartB{}) : lean(One{}, One{}, Plain{}, PartB{});
            }
        }
        // A prefetch distance D < S: warp 0 loads both operands; the whole
        // warp runs the loop (warp-uniform control) and lane 0 issues.
        for (int i = 0; ok && D < S && warp == 0; ++i) {
            Unit w;
            if (!item(i, w)) break;
            const int m0 = w.mb * p.bm + int(rank) * p.a_rows, n0 = w.nb * p.bn + int(rank) * p.b_box_rows;
            for (int kb = w.kb0; kb < w.kb1; ++kb) {
                if (!warp_wait(empty(s), ph ^ 1u, p, abort, 0, issued)) {
                    ok = false;
                    break;
                }
                if (D < S) {
                    if (issued >= D && !warp_wait(empty(sd), phd, p, abort, 0, issued)) {
                        ok = false;
                        break;
                    }
                    if (++sd == S) {
                        sd = 0;
                        if (issued >= D) phd ^= 1u;
                    }
                }
                const bool in_range =
                    check(s < S && (kb * p.bk * 2) % 16 == 0 && kb < p.num_kb && w.mb < (MC ? 2 * p.sched_m : p.tiles_m) &&
                              w.nb < p.tiles_n && int(p.panels) * int(p.a_panel16 << 4) <= int(p.a_slot) &&
                              int(p.panels) * int(p.b_panel16 << 4) <= int(p.b_slot),
                          p, abort, 0, issued);
                if (lane == 0 && in_range) {
                    const uint32_t a_dst = sA + uint32_t(s) * p.a_slot, b_dst = sB + uint32_t(s) * p.b_slot;
                    if constexpr (PAIR) {
                        const uint32_t fb = full_leader + 8u * uint32_t(s);
                        if (rank == 0) mbar_arrive_expect_tx(full(s), p.stage_tx);
                        for (int pl = 0; pl < p.panels; ++pl) {
                            const int x = kb * p.bk + pl * p.panel_k;
                            const uint32_t a_at = a_dst + (uint32_t(pl) * p.a_panel16 << 4);
                            const uint32_t b_at = b_dst + (uint32_t(pl) * p.b_panel16 << 4);
                            // a wide tile's second N-half: this CTA's rows of it, block_N / 2 further on
                            const uint32_t b2_at = b_dst + ((uint32_t(pl) * p.b_panel16 + p.b_half16) << 4);
                            if constexpr (MC) {
                                // B: this CTA's part of its rows, multicast to it and to the CTA of
                                // the other pair that holds the same rows (rank ^ 2)
                                const uint32_t part = pidx ? uint32_t(p.b_part0) * p.row_bytes : 0u;
                                const int yp = pidx ? p.b_part0 : 0;
                                const void *bmap = pidx ? &p.tmB1 : &p.tmB;
                                const uint16_t mask = uint16_t((1u << crank) | (1u << (crank ^ 2u)));
                                if (p.stream_ops) {
                                    tma_load_2d_pair_hint(a_at, &p.tmA, x, m0, fb, policy);
                                    tma_load_2d_pair_mc_hint(b_at + part, bmap, x, n0 + yp, fb, mask, policy);
                                    if (p.n_halves == 2)
                                        tma_load_2d_pair_mc_hint(b2_at + part, bmap, x, n0 + (p.bn >> 1) + yp, fb, mask,
                                                                 policy);
                                } else {
                                    tma_load_2d_pair(a_at, &p.tmA, x, m0, fb);
                                    tma_load_2d_pair_mc(b_at + part, bmap, x, n0 + yp, fb, mask);
                                    if (p.n_halves == 2)
                                        tma_load_2d_pair_mc(b2_at + part, bmap, x, n0 + (p.bn >> 1) + yp, fb, mask);
                                }
                            } else if (p.stream_ops) {
                                tma_load_2d_pair_hint(a_at, &p.tmA, x, m0, fb, policy);
                                tma_load_2d_pair_hint(b_at, &p.tmB, x, n0, fb, policy);
                                if (p.n_halves == 2) tma_load_2d_pair_hint(b2_at, &p.tmB, x, n0 + (p.bn >> 1), fb, policy);
                            } else {
                                tma_load_2d_pair(a_at, &p.tmA, x, m0, fb);
                                tma_load_2d_pair(b_at, &p.tmB, x, n0, fb);
                                if (p.n_halves == 2) tma_load_2d_pair(b2_at, &p.tmB, x, n0 + (p.bn >> 1), fb);
                            }
                        }
                    } else {
                        mbar_arrive_expect_tx(full(s), p.stage_tx);
                        for (int pl = 0; pl < p.panels; ++pl) {
                            const int x = kb * p.bk + pl * p.panel_k;
                            const uint32_t a_at = a_dst + (uint32_t(pl) * p.a_panel16 << 4);
                            const uint32_t b_at = b_dst + (uint32_t(pl) * p.b_panel16 << 4);
                            if (p.stream_ops) {
                                tma_load_2d_hint(a_at, &p.tmA, x, m0, full(s), policy);
                                tma_load_2d_hint(b_at, &p.tmB, x, n0, full(s), policy);
                            } else {
                                tma_load_2d(a_at, &p.tmA, x, m0, full(s));
                                tma_load_2d(b_at, &p.tmB, x, n0, full(s));
                            }
                        }
                    }
                }
                __syncwarp();
                ++issued;
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            // Let the loads still in flight land before the CTA may exit:
            // only the last min(S, issued) slots can be outstanding.  With
            // two producer warps a slot may hold one warp's loads only (the
            // other gave up first), and in mode 3 a CTA's B copies also land in
            // the other pair, whose barriers it cannot wait on: there the
            // fixed wait below.
            if (D < S && !MC && (!PAIR || rank == 0)) {
                const int first = issued > S ? issued - S : 0;
                for (int j = first; j < issued; ++j)
                    wait_bar(full(j % S), uint32_t((j / S) & 1), p, abort, 0, j, false);
            } else {
                // The odd CTA's loads complete the even CTA's barriers, which it
                // cannot wait on (try_wait reads only this CTA's barriers), and
                // the even CTA cannot wait on them either once it has aborted: a
                // phase it never armed does not complete.  So the odd CTA gives
                // its loads a fixed time to land.  At most S slots of at most
                // 64 KB each are outstanding per CTA; even if every SM's ring
                // were in flight at once (152 x 227 KB, about 35 MB) HBM at
                // 6.7 TB/s delivers it in about 5 us, so 2 ms is a margin of
                // several hundred.  This path runs only after a watchdog
                // expiry, when the launch's result is already discarded.
                const uint64_t t0 = globaltimer();
                while (globaltimer() - t0 < 2000000ull) {
                }
            }
        }
        __syncwarp();
        if constexpr (CSPLIT) {  // the two cluster barriers of csplit_epilogue
            cluster_sync();
            cluster_sync();
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: the warp runs the loop, one elected lane drives the tensor core.
        // The k-steps per slot and the MMAs per k-step are compile-time in
        // the issue loop, so each MMA costs one descriptor add.
        if (!PAIR || rank == 0) {
            const uint16_t pm = uint16_t(0x3u << leader);
            const MmaCtx c{sA, sB, tmem, bars, S, stall, drain, unit0, ustride, uint16_t(MC ? 0xFu : 0x3u), pm,
                           uint16_t(0x1u << leader)};
            if (p.mma_per_kstep == 2)
                mma_dispatch_nk<2, PAIR>(p, c, abort, lane);
            else
                mma_dispatch_nk<1, PAIR>(p, c, abort, lane);
        }
        if constexpr (CSPLIT) {  // the two cluster barriers of csplit_epilogue
            __syncwarp();
            cluster_sync();
            cluster_sync();
        }
    } else if constexpr (CSPLIT) {
        csplit_epilogue(p, sA, reinterpret_cast<int *>(smem + p.off_c), tmem, acc_full(0), abort, warp, lane, unit0);
    } else {
        // ---------------- epilogue: 8 warps; warp w reads TMEM lanes 32*(w%4)..+31,
        // and the two warps of a lane quarter take alternate 32-column chunks.
        const int q = warp & 3;
        const int sub = (warp - 2) >> 2;
        const uint32_t lane_base = uint32_t(q * 32) << 16;
        const int nbuf = p.epi_bufs;
        const uint32_t my_bufs = sC + uint32_t((warp - 2) * nbuf) * p.c_buf_bytes;
        int a = 0;
        uint32_t aph = 0;
        uint32_t chunk = 0;
        int tiles_done = 0;
        constexpr int kRanks = PAIR ? 2 : 1;
        // The epilogue warps meet on epi_bar, one arrival per warp.  The wait is
        // bounded: a warp that left the loop on an abort turns into a recorded
        // timeout for the others, never a hang.
        uint32_t epi_ph = 0;
        auto epi_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(epi_bar);
            const bool met = warp_wait(epi_bar, epi_ph, p, abort, 2, tiles_done, false);
            epi_ph ^= 1u;
            return met;
        };
        bool sk_ok = true;
        for (int i = 0;; ++i, ++tiles_done) {
            Unit w;
            if (!item(i, w)) break;
            const int m0 = w.mb * p.bm + int(rank) * p.a_rows, n0 = w.nb * p.bn;
            if (!warp_wait(acc_full(a), aph, p, abort, 2, tiles_done)) break;
            tc_fence_after();
            // A stream-K piece that is not its whole tile: every piece of the tile
            // stores its fp32 partial (pass 1) and counts in; the last to count adds
            // all the tile's pieces in k order (pass 2) and writes C.
            const bool piece = w.sk && !(w.kb0 == 0 && w.kb1 == p.num_kb);
            const int lo = piece ? sk_lo(p, w.sk_tile) : 0;
            const int hi = piece ? sk_hi(p, w.sk_tile) : -1;
            // Piece of worker v in stream-K tile t: workspace slot 2v + (t - first tile of v).
            auto piece_at = [&](int v, int r, int col) -> float * {
                const int j = w.sk_tile - int(sk_start(p, v) / p.num_kb);
                return p.sk_ws + ((int64_t(2 * v + j) * kRanks + int64_t(rank)) * p.sk_rows + r) * p.bn + col;
            };
            // One pass over this warp's chunks.  mode 0: plain epilogue; 1: store
            // this CTA's piece; 2: add the tile's pieces, then the plain epilogue.
            auto chunks = [&](int mode) {
                int idx = 0;
                for (int h = 0; h < p.m_halves; ++h) {
                    // this warp's accumulator rows: quarter_rows of them, from TMEM lane 32q;
                    // with 16 rows (M = 64) lanes 16-31 load and stage values the store leaves out
                    const int row0 = m0 + h * 128 + q * p.quarter_rows;
                    if (row0 >= p.M) continue;  // warp-uniform
                    const int prow = h * 128 + q * p.quarter_rows + lane;  // row within this CTA's part
                    for (int c = 0; c * kEpiCols < p.bn; ++c) {
                        const int col0 = n0 + c * kEpiCols;
                        if (col0 >= p.N) break;  // warp-uniform
                        if ((idx++ & 1) != sub) continue;  // the other warp of this quarter takes it
                        // the chunk's TMEM columns, staging buffer and store box lie inside their regions,
                        // a piece's row and columns inside its workspace slot
                        if (!check(a * p.acc_cols + h * p.bn + (c + 1) * kEpiCols <= p.tmem_cols &&
                                       uint32_t((warp - 1) * nbuf) * p.c_buf_bytes <= p.off_bar - p.off_c &&
                                       col0 % 8 == 0 && w.row_off + row0 >= 0 &&
                                       (mode == 0 || (h * 128 + (q + 1) * p.quarter_rows <= p.sk_rows &&
                                                      w.sk_tile < p.sk_tiles && lo >= 0 && hi < p.workers)),
                                   p, abort, 2, tiles_done))
                            continue;
                        uint32_t v[32];
                        if (p.num_kb > 0) {
                            tmem_ld_32x32b_x32(tmem + lane_base + uint32_t(a * p.acc_cols + h * p.bn + c * kEpiCols),
                                               v);
                            tmem_wait_ld();
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e) v[e] = 0u;  // empty reduction
                        }
                        if (mode == 1) {
                            if (lane < p.quarter_rows) {
                                float4 *dst = reinterpret_cast<float4 *>(piece_at(unit0, prow, c * kEpiCols));
#pragma unroll
                                for (int e = 0; e < 8; ++e)
                                    dst[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                                         __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
                            }
                            continue;
                        }
                        if (mode == 2 && lane < p.quarter_rows) {
                            // the pieces of workers lo .. hi in that (k) order; this CTA's own is v
                            float4 acc[8];
                            for (int vw = lo; vw <= hi; ++vw) {
                                float4 x[8];
                                if (vw == unit0) {
#pragma unroll
                                    for (int e = 0; e < 8; ++e)
                                        x[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                                           __uint_as_float(v[4 * e + 2]),
                                                           __uint_as_float(v[4 * e + 3]));
                                } else {
                                    const float4 *src =
                                        reinterpret_cast<const float4 *>(piece_at(vw, prow, c * kEpiCols));
#pragma unroll
                                    for (int e = 0; e < 8; ++e) x[e] = __ldcg(src + e);
                                }
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    if (vw == lo) {
                                        acc[e] = x[e];
                                    } else {
                                        acc[e].x += x[e].x;
                                        acc[e].y += x[e].y;
                                        acc[e].z += x[e].z;
                                        acc[e].w += x[e].w;
                                    }
                                }
                            }
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                v[4 * e] = __float_as_uint(acc[e].x);
                                v[4 * e + 1] = __float_as_uint(acc[e].y);
                                v[4 * e + 2] = __float_as_uint(acc[e].z);
                                v[4 * e + 3] = __float_as_uint(acc[e].w);
                            }
                        }
                        // Staging: each TMA store box is 32 rows of 64 bytes (32 16-bit or 16 fp32
                        // columns; 64-byte swizzle, 16-byte piece j of row r at j ^ ((r / 2) % 4)) in one
                        // of this warp's two buffers, so a box is staged while the previous box's store
                        // still reads the other buffer.  A 32-column chunk is one box of 16-bit output
                        // and two of fp32.
#pragma unroll
                        for (int bx = 0; bx < 2; ++bx) {
                            const int bcol = col0 + bx * (kEpiCols / 2);
                            if (bx == 1 && (p.out_mode != 0 || bcol >= p.N)) break;  // warp-uniform
                            const uint32_t buf = my_bufs + (chunk & 1u) * p.c_buf_bytes;
                            if (chunk >= 2u && lane == 0) bulk_wait_read<1>();  // its previous store has read it
                            __syncwarp();
                            const uint32_t row = buf + uint32_t(lane) * 64u;
                            if (p.out_mode == 0) {
#pragma unroll
                                for (int j = 0; j < 4; ++j)
                                    st_shared_v4(row + (uint32_t(j ^ ((lane >> 1) & 3)) << 4), v[16 * bx + 4 * j],
                                                 v[16 * bx + 4 * j + 1], v[16 * bx + 4 * j + 2], v[16 * bx + 4 * j + 3]);
                            } else {
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    uint32_t hw[4];
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        const float x0 = __uint_as_float(v[8 * j + 2 * e]);
                                        const float x1 = __uint_as_float(v[8 * j + 2 * e + 1]);
                                        if (p.out_mode == 1) {
                                            __half2 h2 = __floats2half2_rn(x0, x1);
                                            hw[e] = *reinterpret_cast<uint32_t *>(&h2);
                                        } else {
                                            __nv_bfloat162 b2 = __floats2bfloat162_rn(x0, x1);
                                            hw[e] = *reinterpret_cast<uint32_t *>(&b2);
                                        }
                                    }
                                    st_shared_v4(row + (uint32_t(j ^ ((lane >> 1) & 3)) << 4), hw[0], hw[1], hw[2],
                                                 hw[3]);
                                }
                            }
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_2d(&p.tmC, bcol, w.row_off + row0, buf);
                                bulk_commit();
                            }
                            ++chunk;
                        }
                    }
                }
            };
            if (!piece) {
                chunks(0);
            } else {
                chunks(1);
                __threadfence();  // this thread's piece is visible GPU-wide before the count below
                sk_ok = epi_sync();
                if (sk_ok && threadIdx.x == 2 * 32) {
                    int *cnt = p.sk_cnt + w.sk_tile * kRanks + int(rank);
                    const int last = atomicAdd(cnt, 1) == hi - lo;
                    if (last) *cnt = 0;  // every piece of this launch is in: ready for the next launch
                    *flag = last;
                }
                sk_ok = sk_ok && epi_sync();
                if (sk_ok && *reinterpret_cast<volatile int *>(flag)) {
                    __threadfence();
                    chunks(2);
                }
            }
            // All TMEM reads of accumulator a are done: hand it back to the MMA warp.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR)
                    mbar_arrive_cluster(map_to_rank(acc_empty(a), leader));
                else
                    mbar_arrive(acc_empty(a));
            }
            if (++a == p.acc_stages) {
                a = 0;
                aph ^= 1u;
            }
            if (!sk_ok) break;  // the epilogue warps lost step: give up (the timeout is recorded)
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
        if (p.grid_reduce) grid_reduce_phase(p, abort, flag, sA, bulk_bar);
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // neither CTA leaves while the pair's MMAs or arrivals may touch it
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem, uint32_t(p.tmem_cols));
        else
            tmem_dealloc(tmem, uint32_t(p.tmem_cols));
    }
}

// Split-K reduction: C[i] = sum over s = 0, 1, ..., splits-1 (in that order)
// of the fp32 partials W[s * stride + i], rounded once to the output type.
// Elementwise and HBM-bound: four consecutive elements per thread per step
// (M*N and the split stride are multiples of 4 because every row pitch is a
// multiple of 16 bytes).
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float *__restrict__ W, void *__restrict__ C,
                                                            int64_t mn, int64_t stride, int splits, int out_mode)
{
    griddep_wait();  // launched as a programmatic dependent of the GEMM: its partials are complete
    const int64_t n4 = mn / 4;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += int64_t(gridDim.x) * blockDim.x) {
        float4 acc = reinterpret_cast<const float4 *>(W)[i];
        for (int s = 1; s < splits; ++s) {
            const float4 v = reinterpret_cast<const float4 *>(W + int64_t(s) * stride)[i];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        if (out_mode == 0) {
            reinterpret_cast<float4 *>(C)[i] = acc;
        } else if (out_mode == 1) {
            __half2 lo = __floats2half2_rn(acc.x, acc.y), hi = __floats2half2_rn(acc.z, acc.w);
            uint2 u;
            u.x = *reinterpret_cast<uint32_t *>(&lo);
            u.y = *reinterpret_cast<uint32_t *>(&hi);
            reinterpret_cast<uint2 *>(C)[i] = u;
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 u;
            u.x = *reinterpret_cast<uint32_t *>(&lo);
            u.y = *reinterpret_cast<uint32_t *>(&hi);
            reinterpret_cast<uint2 *>(C)[i] = u;
        }
    }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

static CUtensorMapSwizzle swizzle_for(int row_bytes)
{
    return row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
           : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                             : CU_TENSOR_MAP_SWIZZLE_32B;
}

// Descriptor swizzle field (bits 61-63): 128 B -> 2, 64 B -> 4, 32 B -> 6.
static uint32_t desc_layout_for(int row_bytes) { return row_bytes == 128 ? 2u : row_bytes == 64 ? 4u : 6u; }

static CUtensorMapDataType tmap_dtype(int dt)
{
    return dt == kF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
           : dt == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// L2 promotion of the operand loads.  With rows that start on 128-byte
// boundaries, 256-byte promotion helps slightly.  When the row pitch is not a
// multiple of 128 bytes (K = 5000 at 16 bits), every 128-byte box row
// straddles two lines; there 256-byte promotion measured about 5 % slower
// than 128-byte promotion.
static CUtensorMapL2promotion operand_promotion(uint64_t pitch_bytes)
{
    return pitch_bytes % 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
}

static int encode_2d(CUtensorMap *m, int dt, const void *base, uint64_t inner, uint64_t outer, uint64_t pitch_bytes,
                     uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz, CUtensorMapL2promotion l2)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return kErrCuda;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {pitch_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, tmap_dtype(dt), 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? kOk : kErrCuda;
}

}  // namespace tg

using namespace tg;

struct tgemm_plan_s {
    int64_t M, N, K;
    int dtype, out_dtype;
    Layout L;
    int device;
    int num_sms;
    int smem_limit;
    int smem_launch;
    int tiles_m, tiles_n, num_tiles, grid, group_m;
    int pair;  // clusters of two CTAs per block_M = 256 tile
    int mc;    // clusters of two pairs sharing B through multicast (kernel mode 3)
    int splits;                // K splits (1: none)
    int csk;                   // > 1: splits reduced inside the kernel by clusters of csk CTAs
    float *d_work;             // split-K partial sums: splits (or, with csk, splits / csk) x M x N fp32
    int *d_counters;           // csk with more than one cluster per tile: arrival counters
    int grid_reduce;           // K splits reduced in the GEMM kernel after a grid-wide barrier
    uint32_t *d_gbar;          // that barrier's arrival count and generation
    int sk_tiles;              // tiles of the stream-K tail (0: none)
    float *d_sk_ws;            // the tail's partial pieces
    int *d_status;
    unsigned long long watchdog_ns;
    int debug_stall;
    // tensor maps cached for the last pointer triple
    const void *cA, *cB;
    void *cC;
    bool maps_valid;
    Params params;
};

static const unsigned long long kDefaultWatchdogNs = 2000000000ull;

// The kernel's dynamic shared-memory ceiling is a per-function, per-device
// attribute: set it once per device to the device's opt-in limit, so that
// every plan (whatever its own footprint) can launch.
static int allow_max_smem(int dev, int limit)
{
    static std::mutex mu;
    static bool done[64] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && done[dev]) return kOk;
    if (cudaFuncSetAttribute(tgemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, limit) != cudaSuccess ||
        cudaFuncSetAttribute(tgemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, limit) != cudaSuccess ||
        cudaFuncSetAttribute(tgemm_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, limit) != cudaSuccess ||
        cudaFuncSetAttribute(tgemm_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, limit) != cudaSuccess) {
        cudaGetLastError();
        return kErrCuda;
    }
    if (dev >= 0 && dev < 64) done[dev] = true;
    return kOk;
}

// Kernel parameters of a launch configuration (everything but the tensor maps,
// the status record and the watchdog).  pair: CTA pairs; splits: effective K
// splits; prefetch: the producer's lead in k-blocks.
static void fill_params(Params &q, const Layout &L, int64_t M, int64_t N, int64_t K, int dtype, int out_dtype,
                        int block_M, int block_N, int block_K, int num_stages, int pair, int splits, int prefetch,
                        int group_m, int tiles_m, int tiles_n, int workers, int csk = 0)
{
    std::memset(&q, 0, sizeof(q));
    q.M = int(M);
    q.N = int(N);
    q.K = int(K);
    q.num_kb = int((K + block_K - 1) / block_K);
    q.tiles_m = tiles_m;
    q.sched_m = tiles_m;
    q.tiles_n = tiles_n;
    q.num_tiles = tiles_m * tiles_n;
    q.group_m = group_m;
    q.splits = splits;
    // effective_splits guarantees every split a non-empty k-block range
    q.kb_per_split = splits > 1 ? (q.num_kb + splits - 1) / splits : q.num_kb;
    q.prefetch = prefetch;
    q.num_units = q.num_tiles * splits;
    q.split_rows = tiles_m * block_M;
    q.bm = block_M;
    q.bn = block_N;
    q.bk = block_K;
    q.stages = num_stages;
    q.n_kstep = block_K * L.in_bytes / 32;  // one MMA consumes K = 16 elements = 32 bytes
    q.m_halves = L.m_halves;
    q.quarter_rows = L.quarter_rows;
    q.a_rows = L.a_rows;
    q.b_rows = L.b_rows;
    q.n_halves = L.n_halves;
    q.b_box_rows = L.b_rows / L.n_halves;
    q.mma_per_kstep = L.m_halves * L.n_halves;
    // second MMA of a k-step: the lower M-half (128 rows of A further on, block_N
    // accumulator columns further on) or the right N-half (the second group of this
    // CTA's B rows, block_N / 2 columns further on)
    q.acc_step = L.n_halves == 2 ? uint32_t(block_N / 2) : uint32_t(block_N);
    q.a_half16 = L.m_halves == 2 ? (128u * uint32_t(L.swizzle_bytes)) >> 4 : 0u;
    q.b_half16 = L.n_halves == 2 ? (uint32_t(q.b_box_rows) * uint32_t(L.swizzle_bytes)) >> 4 : 0u;
    // The kernel's own output: fp32 partials when K is split and reduced by a
    // second kernel, else C's type.
    q.out_mode = splits > 1 && csk <= 1 ? 0 : out_dtype == kF32 ? 0 : out_dtype == kF16 ? 1 : 2;
    // Persistent schedule: workers take whole units round robin; a plan with a
    // stream-K tail sets dp_units and sk_tiles afterwards.
    q.workers = workers;
    q.dp_units = q.num_units;
    q.sk_tiles = 0;
    q.sk_rows = L.m_halves * 4 * L.quarter_rows;
    q.csk = csk > 1 ? csk : 0;
    q.outer = csk > 1 ? splits / csk : 1;
    q.slice_w = csk > 1 ? block_N / csk : 0;
    q.acc_stages = L.acc_stages;
    q.acc_cols = L.acc_cols;
    q.tmem_cols = L.tmem_cols;
    // Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B
    // format (bits 7-9, 10-12: 0 fp16, 1 bf16), both K-major (bits 15, 16 =
    // 0), N >> 3 (bits 17-22), M >> 4 (bits 24-28): M = 128 for one CTA,
    // M = 256 for the CTA pair.
    const uint32_t ab = dtype == kBF16 ? 1u : 0u;
    const uint32_t mma_m = pair ? 256u : block_M == 64 ? 64u : 128u;
    const uint32_t mma_n = uint32_t(block_N / L.n_halves);
    q.idesc = (1u << 4) | (ab << 7) | (ab << 10) | ((mma_n >> 3) << 17) | ((mma_m >> 4) << 24);
    q.a_slot = round_up(L.a_stage_bytes, kSmemAlign);
    q.b_slot = round_up(L.b_stage_bytes, kSmemAlign);
    // Bytes that complete one full[s] phase: this CTA's boxes, or both CTAs' in pair mode.
    q.stage_tx = (L.a_stage_bytes + L.b_stage_bytes) * (pair ? 2u : 1u);
    q.row_bytes = uint32_t(L.swizzle_bytes);
    q.panels = L.panels;
    q.panel_k = L.swizzle_bytes / L.in_bytes;
    q.a_panel16 = (uint32_t(L.a_rows) * uint32_t(L.swizzle_bytes)) >> 4;
    q.b_panel16 = (uint32_t(L.b_rows) * uint32_t(L.swizzle_bytes)) >> 4;
    q.off_a = L.off_a;
    q.off_b = L.off_b;
    q.off_c = L.off_c;
    q.off_bar = L.off_bar;
    q.c_buf_bytes = L.c_buf_bytes;
    q.epi_bufs = L.epi_bufs;
    // Leading byte offset is unused for swizzled K-major tiles whose K extent
    // per MMA lies inside one swizzle row; encode 16 bytes.  Stride byte
    // offset: 8 rows of one swizzle span each.
    q.desc_lo_flags = (1u << 16);
    const uint32_t sbo = 8u * uint32_t(L.swizzle_bytes);
    q.desc_hi = ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (desc_layout_for(L.swizzle_bytes) << 29);
}

// Tensor maps of A, B and the kernel's output: C, or with split K the
// workspace `work`, viewed as [splits * split_rows, N] fp32.
static int encode_maps(Params &q, const Layout &L, int dtype, int out_dtype, const void *A, const void *B, void *C,
                       float *work)
{
    const uint64_t M = uint64_t(q.M), N = uint64_t(q.N), K = uint64_t(q.K);
    int rc = kOk;
    if (K > 0) {
        const CUtensorMapSwizzle swz = swizzle_for(L.swizzle_bytes);
        const uint32_t box_k = uint32_t(L.swizzle_bytes / L.in_bytes);  // one K-panel per box
        const uint64_t pitch = K * uint64_t(L.in_bytes);
        rc = encode_2d(&q.tmA, dtype, A, K, M, pitch, box_k, uint32_t(L.a_rows), swz, operand_promotion(pitch));
        // mode 3: B comes in two multicast parts, rows [0, b_part0) and [b_part0, b_box_rows)
        const uint32_t b_box = uint32_t(L.b_rows / L.n_halves);
        const uint32_t part0 = q.b_part0 > 0 ? uint32_t(q.b_part0) : b_box;
        if (rc == kOk)
            rc = encode_2d(&q.tmB, dtype, B, K, N, pitch, box_k, part0, swz, operand_promotion(pitch));
        if (rc == kOk && q.b_part0 > 0)
            rc = encode_2d(&q.tmB1, dtype, B, K, N, pitch, box_k, b_box - part0, swz, operand_promotion(pitch));
    }
    if (rc != kOk) return rc;
    // one store box per staging buffer: 64 bytes (32 16-bit or 16 fp32 columns) of one warp's
    // accumulator rows, 64-byte swizzle
    const uint32_t box_rows = uint32_t(L.quarter_rows);
    if (q.splits > 1 && q.csk == 0)
        return encode_2d(&q.tmC, kF32, work, N, uint64_t(q.splits) * uint64_t(q.split_rows), N * 4u,
                         uint32_t(kEpiCols / 2), box_rows, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE);
    return encode_2d(&q.tmC, out_dtype, C, N, M, N * uint64_t(L.out_bytes), uint32_t(64 / L.out_bytes), box_rows,
                     CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

// Ranges of the plan options (NULL: all defaults).
static int check_opts(const tgemm_plan_opts *opts, int num_stages)
{
    if (!opts) return kOk;
    if (opts->cta_pair != 0 && opts->cta_pair != 1) return kErrInvalidArg;
    if (opts->group_m < 0 || opts->group_m > 4096) return kErrInvalidArg;
    if (opts->split_k < 0 || opts->split_k > kMaxSplits) return kErrInvalidArg;
    if (opts->prefetch < 0 || opts->prefetch > num_stages) return kErrInvalidArg;
    if (opts->cluster_k != 0 && opts->cluster_k != 1 && opts->cluster_k != 2 && opts->cluster_k != 4 &&
        opts->cluster_k != 8)
        return kErrInvalidArg;
    if (opts->stream_operands != 0 && opts->stream_operands != 1) return kErrInvalidArg;
    if (opts->grid_reduce != 0 && opts->grid_reduce != 1) return kErrInvalidArg;
    if (opts->stream_k != 0 && opts->stream_k != 1) return kErrInvalidArg;
    if (opts->stream_k && (opts->split_k > 1 || opts->cluster_k > 1)) return kErrInvalidArg;
    if (opts->multicast_b != 0 && opts->multicast_b != 1) return kErrInvalidArg;
    if (opts->multicast_b && (!opts->cta_pair || opts->stream_k || opts->grid_reduce || opts->cluster_k > 1))
        return kErrInvalidArg;
    return kOk;
}

static unsigned long long env_watchdog()
{
    const char *e = std::getenv("TGEMM_WATCHDOG_NS");
    if (e && *e) {
        char *end = nullptr;
        unsigned long long v = std::strtoull(e, &end, 10);
        if (end && *end == '\0' && v > 0) return v;
    }
    return kDefaultWatchdogNs;
}

extern "C" {

int64_t tgemm_smem_bound(int dtype, int block_M, int block_N, int block_K, int num_stages)
{
    if (dtype != kF16 && dtype != kBF16) return -kErrUnsupportedDtype;
    if (block_M <= 0 || block_N <= 0 || block_K <= 0 || num_stages <= 0) return -kErrInvalidArg;
    return int64_t(num_stages) * (int64_t(block_M) * block_K + int64_t(block_K) * block_N) * dtype_bytes(dtype);
}

int64_t tgemm_smem_bytes(int dtype, int out_dtype, int block_M, int block_N, int block_K, int num_stages)
{
    if (dtype != kF16 && dtype != kBF16) return -kErrUnsupportedDtype;
    if (out_dtype != kF32 && out_dtype != dtype) return -kErrUnsupportedDtype;
    if (!tile_supported(block_M, block_N, block_K, dtype_bytes(dtype))) return -kErrNoKernel;
    if (num_stages < 1 || num_stages > 64) return -kErrInvalidArg;
    return int64_t(make_layout(block_M, block_N, block_K, num_stages, dtype, out_dtype).total);
}

int tgemm_smem_limit(void)
{
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return -kErrCuda;
    }
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
        cudaGetLastError();
        return -kErrCuda;
    }
    return v;
}

int tgemm_validate(int64_t M, int64_t N, int64_t K, int dtype, int out_dtype, int block_M, int block_N, int block_K,
                   int num_stages, int64_t smem_limit)
{
    return validate(M, N, K, dtype, out_dtype, block_M, block_N, block_K, num_stages, smem_limit);
}

int tgemm_validate_ex(int64_t M, int64_t N, int64_t K, int dtype, int out_dtype, int block_M, int block_N,
                      int block_K, int num_stages, int64_t smem_limit, const tgemm_plan_opts *opts)
{
    const int rc = check_opts(opts, num_stages);
    if (rc != kOk) return rc;
    return validate(M, N, K, dtype, out_dtype, block_M, block_N, block_K, num_stages, smem_limit,
                    opts ? opts->cta_pair : 0, opts && opts->split_k > 1 ? opts->split_k : 1,
                    opts && opts->cluster_k > 1 ? opts->cluster_k : 0, opts ? opts->multicast_b : 0);
}

int tgemm_plan(tgemm_plan_t *out, int64_t M, int64_t N, int64_t K, int dtype, int out_dtype, int block_M, int block_N,
               int block_K, int num_stages)
{
    return tgemm_plan_ex(out, M, N, K, dtype, out_dtype, block_M, block_N, block_K, num_stages, nullptr);
}

int tgemm_plan_ex(tgemm_plan_t *out, int64_t M, int64_t N, int64_t K, int dtype, int out_dtype, int block_M,
                  int block_N, int block_K, int num_stages, const tgemm_plan_opts *opts)
{
    if (!out) return kErrInvalidArg;
    *out = nullptr;
    const int pair = opts && opts->cta_pair ? 1 : 0;
    if (check_opts(opts, num_stages) != kOk) return kErrInvalidArg;
    const int splits = effective_splits(K, block_K, opts && opts->split_k > 1 ? opts->split_k : 1);
    const int csk = opts && opts->cluster_k > 1 ? opts->cluster_k : 0;
    const int mc = opts && opts->multicast_b ? 1 : 0;
    // Argument checks that need no device come first.
    int rc = validate(M, N, K, dtype, out_dtype, block_M, block_N, block_K, num_stages, INT64_MAX, pair, splits, csk,
                      mc);
    if (rc != kOk) return rc;
    int dev = 0, major = 0, minor = 0, sms = 0, limit = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) ||
        cudaDeviceGetAttribute(&limit, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) ||
        cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) {
        cudaGetLastError();
        return kErrCuda;
    }
    if (major != 10 || minor != 3) return kErrArch;
    rc = validate(M, N, K, dtype, out_dtype, block_M, block_N, block_K, num_stages, limit, pair, splits, csk, mc);
    if (rc != kOk) return rc;

    tgemm_plan_s *p = new (std::nothrow) tgemm_plan_s();
    if (!p) return kErrCuda;
    p->M = M;
    p->N = N;
    p->K = K;
    p->dtype = dtype;
    p->out_dtype = out_dtype;
    // With K splits reduced by a second kernel, the kernel stages fp32 partial
    // tiles and the reduction converts.
    p->L = make_layout(block_M, block_N, block_K, num_stages, dtype, splits > 1 && !csk ? kF32 : out_dtype, pair);
    p->pair = pair;
    p->mc = mc;
    p->splits = splits;
    p->csk = csk;
    p->d_work = nullptr;
    p->d_counters = nullptr;
    p->grid_reduce = splits > 1 && !csk && opts && opts->grid_reduce ? 1 : 0;
    p->d_gbar = nullptr;
    p->sk_tiles = 0;
    p->d_sk_ws = nullptr;
    p->device = dev;
    p->num_sms = sms;
    p->smem_limit = limit;
    // Request more than half of the SM's shared memory so that exactly one
    // CTA is resident per SM: the persistent schedule and the TMEM allocation
    // (up to all 512 columns) both assume it.
    int one_per_sm = per_sm / 2 + 1;
    p->smem_launch = int(p->L.total) > one_per_sm ? int(p->L.total) : one_per_sm;
    if (p->smem_launch > limit) p->smem_launch = limit;
    p->tiles_m = int((M + block_M - 1) / block_M);
    p->tiles_n = int((N + block_N - 1) / block_N);
    p->num_tiles = p->tiles_m * p->tiles_n;
    const int units = p->num_tiles * splits;
    p->grid = units < sms ? units : sms;
    p->group_m = opts && opts->group_m > 0 ? opts->group_m : 8;
    p->watchdog_ns = env_watchdog();
    p->debug_stall = 0;
    p->maps_valid = false;
    if (cudaMalloc(&p->d_status, 4 * sizeof(int)) != cudaSuccess ||
        cudaMemset(p->d_status, 0, 4 * sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        if (p->d_status) cudaFree(p->d_status);
        delete p;
        return kErrCuda;
    }
    if (allow_max_smem(dev, limit) != kOk) {
        cudaFree(p->d_status);
        delete p;
        return kErrCuda;
    }
    if (mc) {
        // Persistent clusters of two pairs, as many as can be resident at once;
        // a cluster's work item is two M-adjacent tiles of one N-block.
        cudaLaunchConfig_t cfg{};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 4;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        const int items = (p->tiles_m + 1) / 2 * p->tiles_n;
        cfg.gridDim = dim3(unsigned(4 * (items < sms / 4 ? items : sms / 4)), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = size_t(p->smem_launch);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, tgemm_kernel<3>, &cfg) != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            cudaFree(p->d_status);
            delete p;
            return kErrCuda;
        }
        p->grid = 4 * (items < clusters ? items : clusters);
    } else if (pair) {
        // Persistent pairs: as many clusters of two as can be resident at once.
        cudaLaunchConfig_t cfg{};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(unsigned(2 * (units < sms / 2 ? units : sms / 2)), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = size_t(p->smem_launch);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, tgemm_kernel<1>, &cfg) != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            cudaFree(p->d_status);
            delete p;
            return kErrCuda;
        }
        p->grid = 2 * (units < clusters ? units : clusters);
    }
    if (csk) {
        // One CTA per work unit (not persistent): clusters of csk never wait on
        // one another, so the grid may take several waves.  At least one
        // cluster must fit.
        cudaLaunchConfig_t cfg{};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = unsigned(csk);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(unsigned(units), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = size_t(p->smem_launch);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, tgemm_kernel<2>, &cfg) != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            cudaFree(p->d_status);
            delete p;
            return kErrCuda;
        }
        p->grid = units;
    }
    if (opts && opts->stream_k) {
        // Stream-K tail: the tiles past the last whole wave of workers, shared out
        // as runs of k-blocks, if each worker gets at least two of them.
        const int workers = pair ? p->grid / 2 : p->grid;
        const int kb = int((K + block_K - 1) / block_K);
        const int rem = p->num_tiles % workers;
        if (rem > 0 && int64_t(rem) * kb >= 2 * int64_t(workers)) p->sk_tiles = rem;
    }
    const int outer = csk ? splits / csk : splits;  // partial sums that go through the workspace
    if (splits > 1 && outer > 1) {
        const size_t bytes = size_t(outer) * size_t(p->tiles_m) * size_t(block_M) * size_t(N) * sizeof(float);
        if (cudaMalloc(&p->d_work, bytes) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(p->d_status);
            delete p;
            return kErrCuda;
        }
    }
    if (p->grid_reduce) {
        if (cudaMalloc(&p->d_gbar, 2 * sizeof(uint32_t)) != cudaSuccess ||
            cudaMemset(p->d_gbar, 0, 2 * sizeof(uint32_t)) != cudaSuccess) {
            cudaGetLastError();
            if (p->d_gbar) cudaFree(p->d_gbar);
            if (p->d_work) cudaFree(p->d_work);
            cudaFree(p->d_status);
            delete p;
            return kErrCuda;
        }
    }
    if (p->sk_tiles) {
        const int workers = pair ? p->grid / 2 : p->grid;
        const size_t rows = size_t(p->L.m_halves) * 4 * size_t(p->L.quarter_rows);
        const size_t ws = size_t(workers) * 2 * (pair ? 2 : 1) * rows * size_t(block_N) * sizeof(float);
        const size_t cnt = size_t(p->sk_tiles) * (pair ? 2 : 1) * sizeof(int);
        if (cudaMalloc(&p->d_sk_ws, ws) != cudaSuccess || cudaMalloc(&p->d_counters, cnt) != cudaSuccess ||
            cudaMemset(p->d_counters, 0, cnt) != cudaSuccess) {
            cudaGetLastError();
            if (p->d_counters) cudaFree(p->d_counters);
            if (p->d_sk_ws) cudaFree(p->d_sk_ws);
            if (p->d_gbar) cudaFree(p->d_gbar);
            if (p->d_work) cudaFree(p->d_work);
            cudaFree(p->d_status);
            delete p;
            return kErrCuda;
        }
    }
    if (csk && outer > 1) {
        const size_t bytes = size_t(p->num_tiles) * size_t(csk) * sizeof(int);
        if (cudaMalloc(&p->d_counters, bytes) != cudaSuccess || cudaMemset(p->d_counters, 0, bytes) != cudaSuccess) {
            cudaGetLastError();
            if (p->d_counters) cudaFree(p->d_counters);
            if (p->d_work) cudaFree(p->d_work);
            cudaFree(p->d_status);
            delete p;
            return kErrCuda;
        }
    }

    Params &q = p->params;
    fill_params(q, p->L, M, N, K, dtype, out_dtype, block_M, block_N, block_K, num_stages, pair, splits,
                opts && opts->prefetch > 0 ? opts->prefetch : num_stages, p->group_m, p->tiles_m, p->tiles_n,
                mc ? p->grid / 4 : pair ? p->grid / 2 : p->grid, csk);
    if (mc) {
        q.sched_m = (p->tiles_m + 1) / 2;
        q.num_units = q.sched_m * p->tiles_n;  // work items: pairs of M-adjacent tiles
        q.b_part0 = mcast_part0(q.b_box_rows);
    }
    q.watchdog_ns = p->watchdog_ns;
    q.status = p->d_status;
    q.ws = p->d_work;
    q.counters = p->d_counters;
    q.dp_units = q.num_units - p->sk_tiles;
    q.sk_tiles = p->sk_tiles;
    q.sk_ws = p->d_sk_ws;
    q.sk_cnt = p->d_counters;
    q.stream_ops = opts && opts->stream_operands ? 1 : 0;
    q.grid_reduce = p->grid_reduce;
    q.grid_bar = p->d_gbar;
    q.out_mode_final = out_dtype == kF32 ? 0 : out_dtype == kF16 ? 1 : 2;
    *out = p;
    return kOk;
}

static int aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

static int prepare_maps(tgemm_plan_s *p, const void *A, const void *B, void *C)
{
    if (p->maps_valid && p->cA == A && p->cB == B && p->cC == C) return kOk;
    const int rc = encode_maps(p->params, p->L, p->dtype, p->out_dtype, A, B, C, p->d_work);
    if (rc != kOk) {
        p->maps_valid = false;
        return rc;
    }
    p->cA = A;
    p->cB = B;
    p->cC = C;
    p->params.C = C;
    p->maps_valid = true;
    return kOk;
}

int tgemm_run(tgemm_plan_t p, const void *A, const void *B, void *C, tgemm_stream_t stream)
{
    if (!p) return kErrInvalidArg;
    if (p->M == 0 || p->N == 0) return kOk;  // empty product: nothing to write
    if (!C || (p->K > 0 && (!A || !B))) return kErrInvalidArg;
    if (!aligned16(C) || (p->K > 0 && (!aligned16(A) || !aligned16(B)))) return kErrAlignment;
    int rc = prepare_maps(p, A, B, C);
    if (rc != kOk) return rc;
    p->params.watchdog_ns = p->watchdog_ns;
    p->params.debug_stall = p->debug_stall;
    if (p->pair || p->csk || p->grid_reduce) {
        // Clusters for CTA pairs and the cluster reduction; a cooperative
        // launch (every CTA resident at once) for the grid-wide reduction.
        cudaLaunchConfig_t cfg{};
        cudaLaunchAttribute attr[3];
        unsigned na = 0;
        if (!p->grid_reduce) {  // see the one-CTA launch below
            attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[na].val.programmaticStreamSerializationAllowed = 1;
            ++na;
        }
        if (p->pair || p->csk) {
            attr[na].id = cudaLaunchAttributeClusterDimension;
            attr[na].val.clusterDim.x = p->csk ? unsigned(p->csk) : p->mc ? 4u : 2u;
            attr[na].val.clusterDim.y = 1;
            attr[na].val.clusterDim.z = 1;
            ++na;
        }
        if (p->grid_reduce) {
            attr[na].id = cudaLaunchAttributeCooperative;
            attr[na].val.cooperative = 1;
            ++na;
        }
        cfg.gridDim = dim3(unsigned(p->grid), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = size_t(p->smem_launch);
        cfg.stream = reinterpret_cast<cudaStream_t>(stream);
        cfg.attrs = attr;
        cfg.numAttrs = na;
        if (cudaLaunchKernelEx(&cfg,
                               p->csk  ? tgemm_kernel<2>
                               : p->mc ? tgemm_kernel<3>
                               : p->pair ? tgemm_kernel<1>
                                         : tgemm_kernel<0>,
                               p->params) != cudaSuccess) {
            cudaGetLastError();
            return kErrCuda;
        }
    } else {
        // A programmatic dependent of the kernel before it in the stream: its
        // launch and set-up overlap that kernel's last CTAs, and it waits in
        // griddepcontrol.wait before it reads A and B or writes C.  (The
        // cooperative launch of the grid-wide reduction keeps the plain order.)
        cudaLaunchConfig_t cfg{};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.gridDim = dim3(unsigned(p->grid), 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = size_t(p->smem_launch);
        cfg.stream = reinterpret_cast<cudaStream_t>(stream);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, tgemm_kernel<0>, p->params) != cudaSuccess) {
            cudaGetLastError();
            return kErrCuda;
        }
    }
    if (p->splits > 1 && !p->csk && !p->grid_reduce) {
        const int64_t mn = p->M * p->N;
        const int64_t n4 = mn / 4;
        int blocks = int((n4 + 255) / 256);
        const int cap = 8 * p->num_sms;
        if (blocks > cap) blocks = cap;
        const int out_mode = p->out_dtype == kF32 ? 0 : p->out_dtype == kF16 ? 1 : 2;
        const int64_t stride = int64_t(p->params.split_rows) * p->N;
        // A programmatic dependent of the GEMM: it is scheduled while the GEMM's
        // CTAs finish and waits in the kernel for the GEMM grid to complete.
        cudaLaunchConfig_t cfg{};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.gridDim = dim3(unsigned(blocks), 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = reinterpret_cast<cudaStream_t>(stream);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, static_cast<const float *>(p->d_work), C, mn, stride,
                               p->splits, out_mode) != cudaSuccess) {
            cudaGetLastError();
            return kErrCuda;
        }
    }
    return kOk;
}

int tgemm_run_host(tgemm_plan_t p, const void *hA, const void *hB, void *hC, void *dA, void *dB, void *dC,
                   tgemm_stream_t stream)
{
    if (!p) return kErrInvalidArg;
    if (p->M == 0 || p->N == 0) return kOk;
    if (!hC || !dC || (p->K > 0 && (!hA || !hB || !dA || !dB))) return kErrInvalidArg;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t a_bytes = size_t(p->M) * size_t(p->K) * p->L.in_bytes;
    const size_t b_bytes = size_t(p->N) * size_t(p->K) * p->L.in_bytes;
    const size_t c_bytes = size_t(p->M) * size_t(p->N) * p->L.out_bytes;
    if (p->K > 0) {
        if (cudaMemcpyAsync(dA, hA, a_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(dB, hB, b_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
            cudaGetLastError();
            return kErrCuda;
        }
    }
    int rc = tgemm_run(p, dA, dB, dC, stream);
    if (rc != kOk) return rc;
    if (cudaMemcpyAsync(hC, dC, c_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) {
        cudaGetLastError();
        return kErrCuda;
    }
    return kOk;
}

int tgemm_status(tgemm_plan_t p, int *detail)
{
    if (!p) return kErrInvalidArg;
    int h[4] = {0, 0, 0, 0};
    if (cudaMemcpy(h, p->d_status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(p->d_status, 0, sizeof(h)) != cudaSuccess) {
        cudaGetLastError();
        return -kErrCuda;
    }
    // A launch that gave up may have left some of the in-kernel split
    // reduction's arrival counters part-way: clear them for the next launch.
    const size_t n_counters = p->sk_tiles ? size_t(p->sk_tiles) * (p->pair ? 2 : 1) : size_t(p->num_tiles) * p->csk;
    if (h[0] != kOk && ((p->d_counters && cudaMemset(p->d_counters, 0, n_counters * sizeof(int)) != cudaSuccess) ||
                        (p->d_gbar && cudaMemset(p->d_gbar, 0, 2 * sizeof(uint32_t)) != cudaSuccess))) {
        cudaGetLastError();
        return -kErrCuda;
    }
    if (detail) std::memcpy(detail, h, sizeof(h));
    return h[0];
}

int tgemm_set_watchdog_ns(tgemm_plan_t p, uint64_t ns)
{
    if (!p) return kErrInvalidArg;
    p->watchdog_ns = ns ? (unsigned long long)ns : env_watchdog();
    return kOk;
}

int tgemm_debug_stall(tgemm_plan_t p, int on)
{
    if (!p) return kErrInvalidArg;
    p->debug_stall = on ? 1 : 0;
    return kOk;
}

int tgemm_get_plan_info(tgemm_plan_t p, tgemm_plan_info *info)
{
    if (!p || !info) return kErrInvalidArg;
    info->M = p->M;
    info->N = p->N;
    info->K = p->K;
    info->dtype = p->dtype;
    info->out_dtype = p->out_dtype;
    info->block_M = p->L.bm;
    info->block_N = p->L.bn;
    info->block_K = p->L.bk;
    info->num_stages = p->L.stages;
    info->tiles_m = p->tiles_m;
    info->tiles_n = p->tiles_n;
    info->num_tiles = p->num_tiles;
    info->grid = p->grid;
    info->threads = kThreads;
    info->num_k_blocks = p->params.num_kb;
    info->acc_stages = p->L.acc_stages;
    info->tmem_columns = p->L.tmem_cols;
    info->smem_bytes = p->smem_launch;
    info->smem_bound = p->L.bound;
    info->smem_limit = p->smem_limit;
    info->num_sms = p->num_sms;
    info->cta_pair = p->pair;
    info->split_k = p->splits;
    info->prefetch = p->params.prefetch;
    info->num_units = p->params.num_units;
    info->cluster_k = p->csk;
    info->stream_operands = p->params.stream_ops;
    info->grid_reduce = p->grid_reduce;
    info->stream_k_tiles = p->sk_tiles;
    info->multicast_b = p->mc;
    return kOk;
}

int tgemm_destroy(tgemm_plan_t p)
{
    if (!p) return kOk;
    int rc = kOk;
    if (p->d_status && cudaFree(p->d_status) != cudaSuccess) {
        cudaGetLastError();
        rc = kErrCuda;
    }
    if (p->d_work && cudaFree(p->d_work) != cudaSuccess) {
        cudaGetLastError();
        rc = kErrCuda;
    }
    if (p->d_counters && cudaFree(p->d_counters) != cudaSuccess) {
        cudaGetLastError();
        rc = kErrCuda;
    }
    if (p->d_gbar && cudaFree(p->d_gbar) != cudaSuccess) {
        cudaGetLastError();
        rc = kErrCuda;
    }
    if (p->d_sk_ws && cudaFree(p->d_sk_ws) != cudaSuccess) {
        cudaGetLastError();
        rc = kErrCuda;
    }
    delete p;
    return rc;
}

const char *tgemm_strerror(int code)
{
    switch (code < 0 ? -code : code) {
    case kOk: return "ok";
    case kErrInvalidArg: return "invalid argument";
    case kErrUnsupportedDtype: return "unsupported dtype (operands fp16/bf16; output fp32 or the operand dtype)";
    case kErrAlignment: return "pointer or row pitch not a multiple of 16 bytes";
    case kErrSmemBudget: return "num_stages x (A tile + B tile) exceeds the per-block shared-memory limit";
    case kErrNoKernel:
        return "tile shape not implemented (block_M 64/128/256, block_N 32..256 step 32, block_K 16/32/64/128; "
               "CTA pairs need block_M 256)";
    case kErrArch: return "device is not compute capability 10.3 (GB300)";
    case kErrCuda: return "CUDA runtime or driver call failed";
    case kErrTimeout: return "a pipeline wait in the kernel exceeded the watchdog limit";
    case kErrCheck: return "an internal bounds or alignment check failed (debug-check build)";
    default: return "unknown status code";
    }
}

}  // extern "C"

// ---------------------------------------------------------------- allocation-free entry point
//
// For callers that cannot allocate device memory: code that runs where
// cudaMalloc is unavailable or must not be called (inside a custom allocator's
// own hooks, in a service that fixes its device footprint at start-up, or in a
// host runtime that hands the library only the buffers it works on).
// tgemm_plan allocates the kernel's status record with cudaMalloc, so such
// callers cannot use it.  tgemm_run_noalloc runs the same kernel with that
// record -- the only global memory the kernel touches besides A, B and C --
// in the file-scope array below, which the CUDA module provides: every GPU
// that loads this library holds these 256 bytes until the process exits.

static constexpr int kNoallocScratchInts = 64;  // 256 bytes; the kernel needs one 4-int record
static __device__ __align__(256) int g_noalloc_scratch[kNoallocScratchInts];
static constexpr size_t kNoallocRecordBytes = 4 * sizeof(int);  // code, role, block, iteration
static_assert(kNoallocRecordBytes <= sizeof(g_noalloc_scratch), "the status record fits the fixed array");

// Set-up with the calling device current: the array's device address and the
// kernel's shared-memory ceiling.  Host code only sees a host-side stand-in for
// the symbol, so the address comes from cudaGetSymbolAddress -- a host-side
// lookup that allocates nothing.  It is looked up on every call rather than
// cached per device ordinal: after cudaDeviceReset, or in another context on
// the same device, the module is loaded again and the array may move.  The
// first call on a device makes the runtime load the module there.
static int noalloc_setup(int dev, int limit, int **scratch)
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
        cudaGetLastError();
        return kErrCuda;
    }
    if (allow_max_smem(dev, limit) != kOk) return kErrCuda;
    *scratch = static_cast<int *>(p);
    return kOk;
}

extern "C" int tgemm_run_noalloc(int64_t M, int64_t N, int64_t K, int dtype, int out_dtype, int block_M, int block_N,
                                 int block_K, int num_stages, const void *A, const void *B, void *C,
                                 tgemm_stream_t stream, int *status)
{
    int rc = validate(M, N, K, dtype, out_dtype, block_M, block_N, block_K, num_stages, INT64_MAX);
    if (rc != kOk) return rc;
    int dev = 0, major = 0, minor = 0, sms = 0, limit = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) ||
        cudaDeviceGetAttribute(&limit, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) ||
        cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) {
        cudaGetLastError();
        return kErrCuda;
    }
    if (major != 10 || minor != 3) return kErrArch;
    rc = validate(M, N, K, dtype, out_dtype, block_M, block_N, block_K, num_stages, limit);
    if (rc != kOk) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (status) {
        // Reading the status back synchronises the stream, which a stream
        // under capture does not allow: such a call must pass status = NULL.
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
            cudaGetLastError();
            return kErrCuda;
        }
        if (cap != cudaStreamCaptureStatusNone) return kErrInvalidArg;
        *status = kOk;
    }
    if (M == 0 || N == 0) return kOk;  // empty product: nothing to write
    if (!C || (K > 0 && (!A || !B))) return kErrInvalidArg;
    if (!aligned16(C) || (K > 0 && (!aligned16(A) || !aligned16(B)))) return kErrAlignment;
    int *scratch = nullptr;
    rc = noalloc_setup(dev, limit, &scratch);
    if (rc != kOk) return rc;

    const Layout L = make_layout(block_M, block_N, block_K, num_stages, dtype, out_dtype);
    const int one_per_sm = per_sm / 2 + 1;
    int smem = int(L.total) > one_per_sm ? int(L.total) : one_per_sm;
    if (smem > limit) smem = limit;
    const int tiles_m = int((M + block_M - 1) / block_M);
    const int tiles_n = int((N + block_N - 1) / block_N);
    const int tiles = tiles_m * tiles_n;
    const int grid = tiles < sms ? tiles : sms;

    Params q;
    fill_params(q, L, M, N, K, dtype, out_dtype, block_M, block_N, block_K, num_stages, 0, 1, num_stages, 8,
                tiles_m, tiles_n, grid);
    q.watchdog_ns = env_watchdog();
    q.status = scratch;
    rc = encode_maps(q, L, dtype, out_dtype, A, B, C, nullptr);
    if (rc != kOk) return rc;

    // The array keeps the previous call's record: clear it before this launch.
    if (cudaMemsetAsync(scratch, 0, kNoallocRecordBytes, s) != cudaSuccess) {
        cudaGetLastError();
        return kErrCuda;
    }
    tgemm_kernel<0><<<grid, kThreads, smem, s>>>(q);
    if (cudaGetLastError() != cudaSuccess) return kErrCuda;
    if (status) {
        int h[4] = {0, 0, 0, 0};
        if (cudaMemcpyAsync(h, scratch, kNoallocRecordBytes, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess) {
            cudaGetLastError();
            return kErrCuda;
        }
        *status = h[0];
    }
    return kOk;
}
