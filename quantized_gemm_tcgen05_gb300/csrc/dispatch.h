// Host-side problem analysis, kernel registry, heuristic, dispatch cache and
// its text serialisation -- the Context / registry / dispatch cache / Measurer
// roles of "InternLM Lmdeploy Gemm Interface" (section Description).
#pragma once
#include <stdint.h>

#include <map>
#include <string>
#include <tuple>
#include <vector>

#include "work_sched.h"

namespace qg {

// Problem families: dense; with operand transforms (U/V scales, int4 B);
// grouped (MoE); grouped with operand transforms (e.g. W4A16 experts).
enum Family : int32_t { FAM_DENSE = 0, FAM_DQ = 1, FAM_GROUPED = 2, FAM_GROUPED_DQ = 3 };

// A validated, normalised problem.  Operand X feeds the UMMA M side (128
// rows per tile), operand Y the N side; which of A / B each one is depends on
// the chosen kernel (swap).
struct Problem {
    int32_t family;
    int64_t M, N, K;
    int32_t batches;
    int32_t a_type, b_type, d_type;
    int32_t kstep;                      // elements per K-step: 64 (16-bit operands) or 128 (8-bit)
    const void* A; int64_t lda, a_bs;
    const void* B; int64_t ldb, b_bs;   // stored N x K (K contiguous); S4: ld in nibbles
    const void* U; int64_t ldu; int32_t u_type, ga;
    const void* V; int64_t ldv, v_bs; int32_t v_type, gb;   // v_bs: grouped, elements between experts
    const void* Z; int64_t ldz, z_bs;                         // int4 zero points (bytes), or null
    const void* C; int64_t ldc, c_bs;
    void* D; int64_t ldd, d_bs;
    float alpha, beta;
    int32_t epi_flags, bias_type; const void* bias;   // fused bias / activation
    const float* qscale; int32_t qzp;                 // int8 D: per-row scale, zero point
    // grouped
    const int32_t* offsets; int32_t num_experts;
};

// A dispatch decision: one registered kernel plus its schedule.
struct Choice {
    int32_t bn = 0;      // UMMA N tile width
    int32_t swap = 0;    // X = B, Y = A (D^T = B^T A^T), for small M
    int32_t sched = 0;   // SchedKind
    int32_t splits = 1;  // split-K slices (SCHED_SPLITK)
    int32_t pair = 0;    // CTA-pair kernel: 256 x bn tiles over clusters of two SMs
    int32_t gemv = 0;    // small-M streaming kernel on the CUDA cores (the fields above unused)
    float us = 0.0f;     // measured time, 0 if never measured
};

struct Key {
    int32_t family, a_type, b_type, d_type, has_c, has_u, has_v, ga, gb;
    int64_t m_bucket, N, K;
    int32_t batches;
    auto tie() const {
        return std::tie(family, a_type, b_type, d_type, has_c, has_u, has_v, ga, gb, m_bucket, N, K, batches);
    }
    bool operator<(const Key& o) const { return tie() < o.tie(); }
};

const std::vector<int32_t>& tuning_seq();
int64_t m_bucket(int64_t M);
Key make_key(const Problem& p);

// Tiles of a problem under a choice, and the schedule parameters.
// sm_count: SMs of the device; the CTA-pair kernel runs on clusters of two.
SchedParams make_sched(const Problem& p, const Choice& c, int sm_count);
size_t partials_bytes_needed(const SchedParams& s, int bn, int pair);
size_t counters_bytes_needed(const SchedParams& s, int pair);

inline bool is_grouped(const Problem& p) { return p.family == FAM_GROUPED || p.family == FAM_GROUPED_DQ; }
inline bool is_dq(const Problem& p) { return p.family == FAM_DQ || p.family == FAM_GROUPED_DQ; }

// Elements per K-step (one 128-byte swizzle row) of the problem's operands.
inline int32_t kstep_of(const Problem& p) { return p.kstep > 0 ? p.kstep : BK_HOST; }

// The small-M streaming kernel takes the problem: M <= 8, one batch, no U
// scale, A 16-bit, B 16-bit or int4 (with or without V).
bool gemv_eligible(const Problem& p);

// Every kernel variant that can run the problem.
std::vector<Choice> candidates(const Problem& p, int sm_count);
// The choice made without measuring.
// allow_gemv: false when the caller asked for a K split (or for none): those
// name schedules of the tensor-core kernels.
Choice heuristic(const Problem& p, int sm_count, size_t partials_bytes, bool allow_gemv = true);
std::string choice_name(const Problem& p, const Choice& c);

// Cache text format (see dispatch.cpp).
std::string cache_serialize(const std::map<Key, Choice>& cache, const std::string& device, int sm, int cc);
bool cache_parse(const std::string& text, const std::string& device, int sm, int cc, std::map<Key, Choice>* out);

}  // namespace qg
