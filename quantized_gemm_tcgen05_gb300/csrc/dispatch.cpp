// Problem analysis, kernel candidates, heuristic and the dispatch-cache text
// format.  Host only.
#include "dispatch.h"

#include <stdlib.h>

#include <math.h>
#include <stdio.h>
#include <string.h>

#include <sstream>

#include "kparams.h"

namespace qg {

const std::vector<int32_t>& tuning_seq() {
    // Batch sizes (M) the dispatch cache is keyed on: dense at small M, where
    // the best kernel changes quickly, then geometric.
    static const std::vector<int32_t> seq = {1,   2,   4,    8,    16,   24,   32,   48,   64,   96,
                                             128, 192, 256,  384,  512,  768,  1024, 1536, 2048, 3072,
                                             4096, 6144, 8192};
    return seq;
}

int64_t m_bucket(int64_t M) {
    for (int32_t v : tuning_seq())
        if (M <= v) return v;
    return ceil_div(M, 8192) * 8192;
}

Key make_key(const Problem& p) {
    Key k;
    k.family = p.family;
    k.a_type = p.a_type;
    k.b_type = p.b_type;
    k.d_type = p.d_type;
    k.has_c = p.beta != 0.0f;
    k.has_u = p.U != nullptr;
    k.has_v = p.V != nullptr;
    k.ga = p.U ? p.ga : 0;
    k.gb = p.V ? p.gb : 0;
    k.m_bucket = m_bucket(p.M);
    k.N = p.N;
    k.K = p.K;
    k.batches = p.batches;
    return k;
}

SchedParams make_sched(const Problem& p, const Choice& c, int sm_count) {
    SchedParams s;
    memset(&s, 0, sizeof s);
    s.k_iters = (int32_t)ceil_div(p.K, kstep_of(p));
    s.batches = p.batches;
    if (is_grouped(p)) {
        // upper bound on padded M-blocks: sum_e ceil(m_e / bm) <= T / bm + E
        // (bm = 256 rows on CTA pairs)
        s.tiles_x = (int32_t)(p.M / (c.pair ? 256 : 128) + p.num_experts);
        s.tiles_y = (int32_t)ceil_div(p.N, c.bn);
        s.batches = 1;
        s.grouped = 1;
        s.expert_offsets = p.offsets;
        s.num_experts = p.num_experts;
    } else if (c.swap) {
        s.tiles_x = (int32_t)ceil_div(p.N, 128);
        s.tiles_y = (int32_t)ceil_div(p.M, c.bn);
    } else {
        s.tiles_x = (int32_t)ceil_div(p.M, c.pair ? 256 : 128);
        s.tiles_y = (int32_t)ceil_div(p.N, c.bn);
    }
    if (c.pair) sm_count /= 2;  // programs are clusters of two CTAs
    const int64_t T = total_tiles(s);
    s.splits = 1;
    s.chunk = s.k_iters;
    s.kind = c.sched;
    if (c.sched == SCHED_SPLITK) {
        int32_t S = c.splits < 1 ? 1 : c.splits;
        if (S > s.k_iters) S = s.k_iters;
        int32_t chunk = (int32_t)ceil_div(s.k_iters, S);
        S = (int32_t)ceil_div(s.k_iters, chunk);
        s.splits = S;
        s.chunk = chunk;
        int64_t units = T * S;
        s.programs = (int32_t)(units < sm_count ? units : sm_count);
        if (S == 1) s.kind = SCHED_DP;
    } else if (c.sched == SCHED_STREAMK) {
        int64_t iters = T * s.k_iters;
        s.programs = (int32_t)(iters < sm_count ? iters : sm_count);
        StreamKPlan pl = streamk_plan((int64_t)s.tiles_x * 128, (int64_t)s.tiles_y * c.bn * s.batches, p.K, 128,
                                      c.bn, kstep_of(p), s.programs);
        s.sk_tiles = (int32_t)pl.streamk_tiles;
        s.sk_full = (int32_t)pl.full_tiles;
        s.sk_partial = (int32_t)pl.partial_tiles;
        s.sk_factor = (int32_t)pl.sm_partition_factor;
        s.sk_maxc = streamk_max_contrib(s.k_iters, s.sk_full);
    } else {
        s.kind = SCHED_DP;
        s.programs = (int32_t)(T < sm_count ? T : sm_count);
    }
    if (s.programs < 1) s.programs = 1;
    return s;
}

// The CTA pair keeps one partial slot and one counter per 128-row half tile.
size_t partials_bytes_needed(const SchedParams& s, int bn, int pair) {
    return (size_t)partial_slots_needed(s) * (pair ? 2 : 1) * 128 * (size_t)bn * sizeof(float);
}

size_t counters_bytes_needed(const SchedParams& s, int pair) {
    if (s.kind == SCHED_DP) return 0;
    return (size_t)total_tiles(s) * (pair ? 2 : 1) * sizeof(int32_t);
}

static int32_t swap_bn(int64_t M) {
    if (M <= 16) return 16;
    if (M <= 32) return 32;
    if (M <= 64) return 64;
    return 128;
}

static bool swap_allowed(const Problem& p) {
    return (p.family == FAM_DENSE || p.family == FAM_DQ) && p.batches == 1 && p.M <= 128;
}

bool gemv_eligible(const Problem& p) {
    if (p.family != FAM_DENSE && p.family != FAM_DQ) return false;
    if (p.batches != 1 || p.M < 1 || p.M > 8 || p.U != nullptr) return false;
    if (p.a_type != DT_F16 && p.a_type != DT_BF16) return false;
    return p.K / 8 < (int64_t(1) << 24);
}

// Largest M the heuristic sends to the streaming kernel (GEMM_GEMV_MAX_M
// overrides the measured default of 2; 0 switches it off).  On GB300 it beats
// the tensor-core decode path at M = 1 (bf16 N 4096 K 14336: 22 vs 26 us;
// W4A16 N 11008 K 4096: 17 vs 27 us), ties at M = 2 and loses from M = 4.
static int64_t gemv_max_m() {
    const char* v = getenv("GEMM_GEMV_MAX_M");
    return v ? atoll(v) : 2;
}

static Choice gemv_choice() {
    Choice c;
    c.bn = 128;  // unused; a valid width keeps cache entries uniform
    c.gemv = 1;
    return c;
}

std::vector<Choice> candidates(const Problem& p, int sm_count) {
    std::vector<Choice> out;
    if (gemv_eligible(p)) out.push_back(gemv_choice());
    const int64_t k_iters = ceil_div(p.K, kstep_of(p));
    auto add_scheds = [&](int32_t bn, int32_t swap) {
        Choice c;
        c.bn = bn;
        c.swap = swap;
        c.sched = SCHED_DP;
        out.push_back(c);
        if (is_grouped(p)) return;
        SchedParams s = make_sched(p, c, sm_count);
        const int64_t T = total_tiles(s);
        if (k_iters >= 2 && T < 4 * (int64_t)sm_count) {
            c.sched = SCHED_STREAMK;
            out.push_back(c);
        }
        if (T < sm_count) {
            const int32_t one_wave = (int32_t)(sm_count / T);
            const bool extra = one_wave != 2 && one_wave != 4 && one_wave != 8;
            for (int32_t S : {2, 4, 8, extra ? one_wave : 0}) {
                if (S < 2 || S > 16 || k_iters < 2 * S) continue;
                c.sched = SCHED_SPLITK;
                c.splits = S;
                out.push_back(c);
            }
        }
    };
    if (is_dq(p)) {
        for (int32_t bn : {64, 128, 256})
            if (bn == 64 || p.N > bn / 2) add_scheds(bn, 0);
        if (swap_allowed(p)) add_scheds(swap_bn(p.M), 1);
        return out;
    }
    add_scheds(128, 0);
    if (p.N > 128)
        for (int32_t bn : {192, 224, 256}) add_scheds(bn, 0);
    if (swap_allowed(p)) add_scheds(swap_bn(p.M), 1);
    if (p.family == FAM_DENSE && p.M > 128)
        for (int32_t bn : {128, 224, 256})
            for (int32_t sched : {SCHED_DP, SCHED_STREAMK}) {
                Choice c;
                c.bn = bn;
                c.pair = 1;
                c.sched = sched;
                out.push_back(c);
            }
    if (p.family == FAM_GROUPED && p.M > 128)
        for (int32_t bn : {224, 256}) {
            Choice c;
            c.bn = bn;
            c.pair = 1;
            out.push_back(c);
        }
    return out;
}

Choice heuristic(const Problem& p, int sm_count, size_t partials_bytes, bool allow_gemv) {
    // Measured on GB300 (152 SMs): full-width 128 x 256 tiles win whenever
    // there are at least as many tiles as SMs; below that, K is split so all
    // SMs stream -- into as many equal slices as fill one wave (split-K),
    // else by stream-K.
    if (allow_gemv && gemv_eligible(p) && p.M <= gemv_max_m()) return gemv_choice();
    Choice c;
    if (swap_allowed(p) && p.M <= 64) {
        c.swap = 1;
        c.bn = swap_bn(p.M);
    } else if (is_dq(p) || p.N <= 128) {
        c.bn = 128;
    } else if (p.family == FAM_GROUPED) {
        // 256-row expert blocks on CTA pairs once they fill a wave of clusters
        // (the tile count is an upper bound; blocks past an expert's rows are
        // skipped), else single-CTA 128 x 256 tiles
        c.bn = 256;
        Choice t = c;
        t.pair = 1;
        if (p.M > 128 && total_tiles(make_sched(p, t, sm_count)) >= sm_count / 2) c.pair = 1;
    } else {
        // the tile shape that minimises waves x time per wave.  Per-wave
        // times measured on GB300 at K = 4096 (64-wide K-steps, two per copy
        // on pairs): CTA pair 15.6 + 0.032*bn us for 256 x bn tiles; single
        // CTA 13.3 + 0.054*bn us for 128 x bn tiles.  Pairs need a full wave
        // of clusters.
        double best = -1.0;
        int32_t best_sched = SCHED_DP;
        for (int32_t pair : {1, 0}) {
            if (pair && (p.family != FAM_DENSE || p.M <= 128)) continue;
            const int64_t cap = pair ? sm_count / 2 : sm_count;
            for (int32_t bn : {256, 224, 192, 128}) {
                if (pair && bn == 192) continue;
                Choice t;
                t.bn = bn;
                t.pair = pair;
                const int64_t T = total_tiles(make_sched(p, t, sm_count));
                if (pair && T < cap) continue;
                const double wave = pair ? 15.6 + 0.032 * bn : 13.3 + 0.054 * bn;
                const double cost = (double)ceil_div(T, cap) * wave;
                if (best < 0 || cost < best - 1e-9) {
                    best = cost;
                    c.bn = bn;
                    c.pair = pair;
                    best_sched = SCHED_DP;
                }
                // stream-K over the pairs evens out a ragged last wave, at the
                // price of partial tiles (measured: about half a wave for the
                // plan's stream-K tiles), where the caller's workspace holds
                // the partials
                if (pair) {
                    t.sched = SCHED_STREAMK;
                    const SchedParams sk = make_sched(p, t, sm_count);
                    const double sk_cost = ((double)T / cap + 0.5) * wave;
                    if (partials_bytes_needed(sk, bn, 1) <= partials_bytes && sk_cost < best - 1e-9) {
                        best = sk_cost;
                        c.bn = bn;
                        c.pair = 1;
                        best_sched = SCHED_STREAMK;
                    }
                }
            }
        }
        if (c.pair) {  // pairs run data-parallel or stream-K (never split-K)
            c.sched = best_sched;
            return c;
        }
    }
    c.sched = SCHED_DP;
    if (is_grouped(p)) return c;
    SchedParams s = make_sched(p, c, sm_count);
    const int64_t T = total_tiles(s);
    const int64_t k_iters = s.k_iters;
    if (T >= sm_count || k_iters < 4) return c;
    const int64_t S = sm_count / T;
    if (S >= 2) {
        c.sched = SCHED_SPLITK;
        c.splits = (int32_t)(S > 8 ? 8 : S);
    } else {
        c.sched = SCHED_STREAMK;
    }
    return c;
}

std::string choice_name(const Problem& p, const Choice& c) {
    if (c.gemv) return "gemv";
    char buf[96];
    const char* fam = p.family == FAM_DQ
                          ? "umma_dq"
                          : (p.family == FAM_GROUPED_DQ
                                 ? "umma_dq_grouped"
                                 : (p.family == FAM_GROUPED ? (c.pair ? "umma2_grouped" : "umma_grouped")
                                                            : (c.pair ? "umma2" : "umma")));
    const char* sk = c.sched == SCHED_DP ? "dp" : (c.sched == SCHED_STREAMK ? "streamk" : "splitk");
    if (c.sched == SCHED_SPLITK)
        snprintf(buf, sizeof buf, "%s_bn%d%s/%s%d", fam, c.bn, c.swap ? "_swap" : "", sk, c.splits);
    else
        snprintf(buf, sizeof buf, "%s_bn%d%s/%s", fam, c.bn, c.swap ? "_swap" : "", sk);
    return buf;
}

// ---- cache text format ------------------------------------------------------------
//
//   qgemm-dispatch-cache 3
//   device <name, spaces as '_'> sm <count> cc <major*10+minor>
//   entries <n>
//   <family> <a> <b> <d> <has_c> <has_u> <has_v> <ga> <gb> <m_bucket> <N> <K> <batches> : <bn> <swap> <sched> <splits> <pair> <gemv> <us>
//   ...
//   end

static std::string sanitize(const std::string& s) {
    std::string r = s;
    for (char& ch : r)
        if (ch == ' ' || ch == '\t' || ch == '\n') ch = '_';
    return r.empty() ? "unknown" : r;
}

std::string cache_serialize(const std::map<Key, Choice>& cache, const std::string& device, int sm, int cc) {
    std::ostringstream os;
    os << "qgemm-dispatch-cache 3\n";
    os << "device " << sanitize(device) << " sm " << sm << " cc " << cc << "\n";
    os << "entries " << cache.size() << "\n";
    for (const auto& kv : cache) {
        const Key& k = kv.first;
        const Choice& c = kv.second;
        char us[32];
        snprintf(us, sizeof us, "%.3f", c.us);
        os << k.family << ' ' << k.a_type << ' ' << k.b_type << ' ' << k.d_type << ' ' << k.has_c << ' ' << k.has_u
           << ' ' << k.has_v << ' ' << k.ga << ' ' << k.gb << ' ' << k.m_bucket << ' ' << k.N << ' ' << k.K << ' '
           << k.batches << " : " << c.bn << ' ' << c.swap << ' ' << c.sched << ' ' << c.splits << ' ' << c.pair << ' '
           << c.gemv << ' ' << us
           << "\n";
    }
    os << "end\n";
    return os.str();
}

static bool valid_choice(const Key& k, const Choice& c) {
    const bool bn_ok = c.bn == 16 || c.bn == 32 || c.bn == 64 || c.bn == 128 || c.bn == 192 || c.bn == 224 || c.bn == 256;
    if (!bn_ok || (c.swap != 0 && c.swap != 1) || c.sched < SCHED_DP || c.sched > SCHED_STREAMK) return false;
    if (c.splits < 1 || c.splits > 64 || !(c.us >= 0.0f)) return false;
    if (c.pair != 0 && c.pair != 1) return false;
    if (c.gemv != 0 && c.gemv != 1) return false;
    if (c.gemv && (c.pair || c.swap || (k.family != FAM_DENSE && k.family != FAM_DQ) || k.m_bucket > 8 || k.has_u))
        return false;
    if (c.pair && (c.swap || c.sched == SCHED_SPLITK || (k.family != FAM_DENSE && k.family != FAM_GROUPED))) return false;
    if (c.pair && c.bn != 128 && c.bn != 224 && c.bn != 256) return false;
    if (k.family < FAM_DENSE || k.family > FAM_GROUPED_DQ) return false;
    if (k.N < 0 || k.K < 0 || k.m_bucket < 1 || k.batches < 1) return false;
    return true;
}

bool cache_parse(const std::string& text, const std::string& device, int sm, int cc, std::map<Key, Choice>* out) {
    std::istringstream is(text);
    std::string magic, word, dev;
    int version = 0, sm_in = -1, cc_in = -1;
    long long n = -1;
    if (!(is >> magic >> version) || magic != "qgemm-dispatch-cache" || version != 3) return false;
    if (!(is >> word) || word != "device" || !(is >> dev)) return false;
    if (!(is >> word) || word != "sm" || !(is >> sm_in)) return false;
    if (!(is >> word) || word != "cc" || !(is >> cc_in)) return false;
    if (dev != sanitize(device) || sm_in != sm || cc_in != cc) return false;
    if (!(is >> word) || word != "entries" || !(is >> n) || n < 0 || n > 1000000) return false;
    std::map<Key, Choice> tmp;
    for (long long i = 0; i < n; ++i) {
        Key k;
        Choice c;
        std::string colon;
        long long mb, N, K;
        if (!(is >> k.family >> k.a_type >> k.b_type >> k.d_type >> k.has_c >> k.has_u >> k.has_v >> k.ga >> k.gb >>
              mb >> N >> K >> k.batches >> colon >> c.bn >> c.swap >> c.sched >> c.splits >> c.pair >> c.gemv >> c.us))
            return false;
        if (colon != ":") return false;
        k.m_bucket = mb;
        k.N = N;
        k.K = K;
        if (!valid_choice(k, c)) return false;
        tmp[k] = c;
    }
    if (!(is >> word) || word != "end") return false;
    for (const auto& kv : tmp) (*out)[kv.first] = kv.second;
    return true;
}

}  // namespace qg
