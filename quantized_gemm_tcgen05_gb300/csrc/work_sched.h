// Work decomposition shared by the host planner and the device kernels.
//
// A GEMM is cut into output tiles (128 rows of the UMMA "M" operand x BN
// columns of the UMMA "N" operand, per batch) and each tile's K range into
// 64-wide steps.  A *unit* is one contiguous run of K-steps of one tile that
// one CTA executes.  Three schedules produce the units:
//
//  * data-parallel: one unit per tile, tiles strided over the persistent grid;
//  * split-K: each tile's K-steps cut into S slices of ceil(k_iters / S) steps
//    (TileLang tutorial "gemm_variants.py", section gemm_splitk, with the
//    remainder kept rather than dropped);
//  * stream-K: the plan of the same page's section streamk_plan; the first
//    streamk_tiles tiles are shared out by iteration across the programs, the
//    rest are handed out whole (section gemm_streamk).
//
// The grouped (MoE) tile map of section gemm_grouped is here too.  Everything
// in this header is plain integer arithmetic compiled for host and device, so
// the host tests check the very code the kernels run.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define QG_HD __host__ __device__ __forceinline__
#else
#define QG_HD inline
#endif

namespace qg {

// A K-step is one 128-byte swizzle row of each operand: 64 16-bit values
// (the default), or 128 8-bit ones.
constexpr int32_t BK_HOST = 64;

enum SchedKind : int32_t { SCHED_DP = 0, SCHED_SPLITK = 1, SCHED_STREAMK = 2 };

struct StreamKPlan {
    int64_t iters_per_tile, total_tiles, streamk_tiles, blocking_tiles, full_tiles, partial_tiles,
        sm_partition_factor;
};

QG_HD int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

QG_HD StreamKPlan streamk_plan(int64_t m, int64_t n, int64_t k, int64_t bm, int64_t bn, int64_t bk,
                               int64_t total_sm) {
    StreamKPlan p;
    p.iters_per_tile = ceil_div(k, bk);
    p.total_tiles = ceil_div(m, bm) * ceil_div(n, bn);
    p.streamk_tiles = p.total_tiles % total_sm;
    if (p.total_tiles - p.streamk_tiles > total_sm) p.streamk_tiles += total_sm;
    p.blocking_tiles = p.total_tiles - p.streamk_tiles;
    int64_t sk_iters = p.streamk_tiles * p.iters_per_tile;
    p.full_tiles = sk_iters / total_sm;
    p.partial_tiles = sk_iters % total_sm;
    int64_t f = p.blocking_tiles / total_sm;
    p.sm_partition_factor = f > 1 ? f : 1;
    return p;
}

// Grouped tile map: padded M-block b -> (expert, first row, rows).  padded
// offsets are the prefix sums of ceil(m_e / bm) * bm; the block belongs to the
// last expert whose padded offset is <= b*bm (zero-row experts share their
// padded offset with the next one, and the later one wins).
QG_HD void grouped_block(const int32_t* off, int32_t E, int32_t bm, int64_t b, int32_t* expert,
                         int64_t* m_start, int32_t* rows) {
    int64_t ms = b * bm, padded = 0, sel_padded = 0;
    int32_t sel = 0;
    for (int32_t i = 0; i < E; ++i) {
        if (ms >= padded) {
            sel = i;
            sel_padded = padded;
        }
        int64_t sz = (int64_t)off[i + 1] - off[i];
        padded += ceil_div(sz, bm) * bm;
    }
    int64_t r = ((int64_t)off[sel + 1] - off[sel]) + sel_padded - ms;
    *expert = sel;
    *m_start = ms - sel_padded + off[sel];
    *rows = (int32_t)(r < 0 ? 0 : (r > bm ? bm : r));
}

// Parameters of one launch's schedule (passed by value to the kernel).
struct SchedParams {
    int32_t kind;       // SchedKind
    int32_t tiles_x;    // tiles along the UMMA M operand (128 rows each)
    int32_t tiles_y;    // tiles along the UMMA N operand (BN rows each)
    int32_t batches;    // independent problems (batched GEMM); 1 otherwise
    int32_t k_iters;    // K-steps per tile
    int32_t splits;     // split-K slices (effective), 1 otherwise
    int32_t chunk;      // split-K steps per slice
    int32_t programs;   // persistent grid size
    // stream-K plan (SCHED_STREAMK)
    int32_t sk_tiles, sk_full, sk_partial, sk_factor;
    int32_t sk_maxc;    // most programs one stream-K tile can have (partial slots per tile)
    // grouped GEMM: device offsets [E+1]; tiles_x is an upper bound then
    const int32_t* expert_offsets;
    int32_t num_experts;
    int32_t grouped;
};

QG_HD int64_t total_tiles(const SchedParams& s) {
    return (int64_t)s.tiles_x * s.tiles_y * s.batches;
}

// What a unit's epilogue does with its accumulator.
enum UnitMode : int32_t { UNIT_FULL = 0, UNIT_PARTIAL = 1 };

struct Unit {
    int64_t tile;      // linear tile id (batch-major, then y, then x)
    int32_t k_begin, k_end;
    int32_t mode;      // UnitMode
    int32_t slot;      // partial slot of this unit (PARTIAL)
    int32_t ncontrib;  // units that contribute to this tile (PARTIAL)
    // coordinates
    int32_t batch;     // batch index, or expert for grouped
    int64_t x_row0;    // first row of the UMMA-M operand (token row for grouped)
    int32_t x_rows;    // valid rows in this tile (grouped masks; else tile height)
    int64_t y_row0;    // first row of the UMMA-N operand
};

// Program that owns stream-K iteration `it` (programs 0..partial-1 run
// full+1 iterations, the rest run full).
QG_HD int64_t streamk_owner(const SchedParams& s, int64_t it) {
    int64_t big = (int64_t)s.sk_partial * (s.sk_full + 1);
    if (it < big) return it / (s.sk_full + 1);
    return s.sk_partial + (it - big) / s.sk_full;
}
QG_HD int64_t streamk_start(const SchedParams& s, int64_t pid) {
    return pid * s.sk_full + (pid < s.sk_partial ? pid : s.sk_partial);
}

// Partial slot of contributor `idx` (0-based, in K order) of tile `tile`.
// Split-K: tile * splits + idx.  Stream-K: each program owns two slots, the
// first for the tile its range starts in and the second for the tile it ends
// in.
// Partial slot of contributor idx (in K order) of a split tile.  Stream-K
// partial units only occur in the plan's stream-K tiles (the first sk_tiles),
// each with at most sk_maxc contributors.
QG_HD int64_t partial_slot(const SchedParams& s, int64_t tile, int32_t idx) {
    if (s.kind == SCHED_SPLITK) return tile * s.splits + idx;
    return tile * s.sk_maxc + idx;
}

QG_HD int64_t partial_slots_needed(const SchedParams& s) {
    if (s.kind == SCHED_SPLITK && s.splits > 1) return total_tiles(s) * s.splits;
    if (s.kind == SCHED_STREAMK) {
        // programs of equal, whole-tile iteration ranges leave no partial tile
        if (s.sk_partial == 0 && s.k_iters > 0 && s.sk_full % s.k_iters == 0) return 0;
        return (int64_t)s.sk_tiles * s.sk_maxc;
    }
    return 0;
}

// Contributors a stream-K tile can have: its k_iters iterations meet at most
// ceil(k_iters / fewest iterations of a program) + 1 programs.
QG_HD int32_t streamk_max_contrib(int32_t k_iters, int32_t sk_full) {
    if (sk_full < 1) return 1;
    return (k_iters + sk_full - 1) / sk_full + 1;
}

// Fill the coordinates of tile `t`.
QG_HD bool tile_coords(const SchedParams& s, int64_t t, Unit& u, int32_t bm, int32_t bn) {
    int64_t per_batch = (int64_t)s.tiles_x * s.tiles_y;
    int64_t b = t / per_batch, r = t % per_batch;
    int64_t tx = r % s.tiles_x, ty = r / s.tiles_x;
    u.tile = t;
    u.y_row0 = ty * bn;
    if (s.grouped) {
        int32_t e, rows;
        int64_t m0;
        grouped_block(s.expert_offsets, s.num_experts, bm, tx, &e, &m0, &rows);
        u.batch = e;
        u.x_row0 = m0;
        u.x_rows = rows;
        return rows > 0;
    }
    u.batch = (int32_t)b;
    u.x_row0 = tx * bm;
    u.x_rows = bm;
    return true;
}

// Per-program iterator over units.  All warp roles of a CTA run their own
// copy and see the same sequence.
struct WorkIter {
    int64_t u;      // DP / split-K: linear unit index
    int64_t it;     // stream-K: next iteration
    int64_t last;   // stream-K: end of this program's iteration range
    int32_t phase;  // stream-K: 0 iterations, 1 blocking tiles
    int32_t p;      // stream-K: blocking index

    QG_HD void init(const SchedParams& s, int32_t pid) {
        u = pid;
        it = 0;
        last = 0;
        phase = 0;
        p = 0;
        if (s.kind == SCHED_STREAMK) {
            it = streamk_start(s, pid);
            last = streamk_start(s, pid + 1);
        }
    }

    QG_HD bool next(const SchedParams& s, int32_t pid, int32_t bm, int32_t bn, Unit& out) {
        const int64_t T = total_tiles(s);
        if (s.kind == SCHED_DP) {
            while (u < T) {
                int64_t t = u;
                u += s.programs;
                if (tile_coords(s, t, out, bm, bn)) {
                    out.k_begin = 0;
                    out.k_end = s.k_iters;
                    out.mode = UNIT_FULL;
                    out.slot = 0;
                    out.ncontrib = 1;
                    return true;
                }
            }
            return false;
        }
        if (s.kind == SCHED_SPLITK) {
            while (u < T * s.splits) {
                int64_t t = u / s.splits;
                int32_t sl = (int32_t)(u % s.splits);
                u += s.programs;
                if (!tile_coords(s, t, out, bm, bn)) continue;
                out.k_begin = sl * s.chunk;
                out.k_end = out.k_begin + s.chunk < s.k_iters ? out.k_begin + s.chunk : s.k_iters;
                out.mode = s.splits > 1 ? UNIT_PARTIAL : UNIT_FULL;
                out.slot = (int32_t)(t * s.splits + sl);
                out.ncontrib = s.splits;
                return true;
            }
            return false;
        }
        // stream-K
        const int64_t ipt = s.k_iters;
        if (phase == 0) {
            if (it < last) {
                int64_t t = it / ipt;
                int64_t kb = it % ipt;
                int64_t end = it + (ipt - kb);
                if (end > last) end = last;
                tile_coords(s, t, out, bm, bn);
                out.k_begin = (int32_t)kb;
                out.k_end = (int32_t)(kb + (end - it));
                if (out.k_begin == 0 && out.k_end == ipt) {
                    out.mode = UNIT_FULL;
                    out.slot = 0;
                    out.ncontrib = 1;
                } else {
                    out.mode = UNIT_PARTIAL;
                    int64_t q0 = streamk_owner(s, t * ipt);
                    int64_t q1 = streamk_owner(s, (t + 1) * ipt - 1);
                    out.slot = (int32_t)partial_slot(s, t, (int32_t)(pid - q0));
                    out.ncontrib = (int32_t)(q1 - q0 + 1);
                }
                it = end;
                return true;
            }
            phase = 1;
        }
        while (p < s.sk_factor) {
            int64_t t = (int64_t)pid + s.sk_tiles + (int64_t)p * s.programs;
            ++p;
            if (t >= T) continue;  // the plan keeps factor >= 1 even with no blocking tile
            tile_coords(s, t, out, bm, bn);
            out.k_begin = 0;
            out.k_end = (int32_t)ipt;
            out.mode = UNIT_FULL;
            out.slot = 0;
            out.ncontrib = 1;
            return true;
        }
        return false;
    }
};

}  // namespace qg
