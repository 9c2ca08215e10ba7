// fused_plan.cuh -- the work list of the fused forward kernel (ssd_fused.cu): how the
// sequences of two-head pairs are cut into super-chunks, and which work item each ticket
// of the kernel's atomic counter stands for.  The decoder is shared by the host planner
// (which simulates the schedule) and the kernel, so both read the list the same way.
#pragma once

#include <stdint.h>

#include <algorithm>
#include <functional>
#include <queue>
#include <vector>

namespace ssd {

// Pair p holds the sequences (b * nh + h) 2p and 2p + 1: two heads of one B/C group.
// Each sequence is ceil(L / 128) sub-chunks of 128 tokens long.  Pairs [0, split) are cut
// into super-chunks of R0 sub-chunks (nsup0 per sequence), the others into super-chunks of
// R1 (nsup1).  A pair cut into nsup > 1 super-chunks needs, for super-chunks 1 .. nsup-1,
// the state entering them: STATE items compute the state each super-chunk 0 .. nsup-2
// produces from a zero start, PASS items chain those states (each PASS item one slice of
// the H x S state columns), and SCAN items walk one super-chunk with the state on chip,
// writing y (and h_final from the last one).
//
// Ticket order: [STATE part 0 | STATE part 1 | PASS | SCAN part 0 | SCAN part 1].  A PASS
// item waits for every STATE item of its pair, a SCAN item of super-chunk m >= 1 for every
// PASS item of its pair; both wait only on items of lower tickets, which running CTAs have
// already taken, so the waits always end.  Within a part, items run super-chunk-major with
// the pairs fastest (the pairs of one B/C group are next to each other).
struct FusedPlan {
    int npair;            // two-head pairs (B * nh / 2)
    int nsub;             // 128-token sub-chunks per sequence
    int split;            // pairs of part 0
    int R0, nsup0;        // part 0: sub-chunks per super-chunk, super-chunks per sequence
    int R1, nsup1;        // part 1
    int nslice;           // PASS slices per cut pair
    int n_state0, n_state1, n_pass, n_scan0, n_scan1, n_items;
    long long sbase1;     // state slot of part 1's first sequence
};

enum FusedKind { kItemState = 0, kItemPass = 1, kItemScan = 2 };

struct FusedItem {
    int kind;
    int pair;             // pair index (sequences 2 pair, 2 pair + 1)
    int m;                // super-chunk (STATE, SCAN)
    int nsup;             // super-chunks per sequence of the pair's part
    int sub_begin;        // first sub-chunk of the super-chunk (STATE, SCAN)
    int nq;               // sub-chunks of the item (0 for PASS)
    int slice;            // PASS slice
    long long slot;       // state slot of super-chunk m of head A (head B: slot + nsup); PASS: slot of m = 0
};

__host__ __device__ inline int fused_cut0(const FusedPlan &p) { return p.nsup0 > 1 ? p.split : 0; }
__host__ __device__ inline int fused_cut1(const FusedPlan &p) { return p.nsup1 > 1 ? p.npair - p.split : 0; }

// Fill the item counts of a plan whose cut (npair, nsub, split, R0, R1, nslice) is set.
__host__ __device__ inline void fused_finish(FusedPlan &p)
{
    p.nsup0 = (p.nsub + p.R0 - 1) / p.R0;
    p.nsup1 = (p.nsub + p.R1 - 1) / p.R1;
    p.n_state0 = fused_cut0(p) * (p.nsup0 - 1);
    p.n_state1 = fused_cut1(p) * (p.nsup1 - 1);
    p.n_pass = (fused_cut0(p) + fused_cut1(p)) * p.nslice;
    p.n_scan0 = p.split * p.nsup0;
    p.n_scan1 = (p.npair - p.split) * p.nsup1;
    p.n_items = p.n_state0 + p.n_state1 + p.n_pass + p.n_scan0 + p.n_scan1;
    p.sbase1 = 2LL * p.split * p.nsup0;
}

__host__ __device__ inline FusedItem fused_item(const FusedPlan &p, int t)
{
    FusedItem it;
    it.slice = 0;
    int part1;
    const int n_state = p.n_state0 + p.n_state1;
    if (t < n_state) {
        it.kind = kItemState;
        part1 = t >= p.n_state0;
        const int i = part1 ? t - p.n_state0 : t;
        const int np = part1 ? p.npair - p.split : p.split;
        it.m = i / np;
        it.pair = (part1 ? p.split : 0) + i % np;
    } else if (t < n_state + p.n_pass) {
        it.kind = kItemPass;
        const int i = t - n_state, ncut0 = fused_cut0(p), ncut = ncut0 + fused_cut1(p);
        it.slice = i / ncut;
        const int c = i % ncut;
        part1 = c >= ncut0;
        it.pair = part1 ? p.split + (c - ncut0) : c;
        it.m = 0;
    } else {
        it.kind = kItemScan;
        const int i0 = t - n_state - p.n_pass;
        part1 = i0 >= p.n_scan0;
        const int i = part1 ? i0 - p.n_scan0 : i0;
        const int np = part1 ? p.npair - p.split : p.split;
        it.m = i / np;
        it.pair = (part1 ? p.split : 0) + i % np;
    }
    const int R = part1 ? p.R1 : p.R0;
    it.nsup = part1 ? p.nsup1 : p.nsup0;
    it.sub_begin = it.m * R;
    const int left = p.nsub - it.sub_begin;
    it.nq = it.kind == kItemPass ? 0 : (left < R ? left : R);
    const long long seqA = part1 ? 2LL * (it.pair - p.split) : 2LL * it.pair;
    it.slot = (part1 ? p.sbase1 : 0) + seqA * it.nsup + it.m;
    return it;
}

// ---- host-side planner (host-only functions) ---------------------------------------------

inline FusedPlan fused_candidate(int npair, int nsub, int split, int R0, int R1, int nslice)
{
    FusedPlan p = {};
    p.npair = npair;
    p.nsub = nsub;
    p.split = split;
    p.R0 = R0;
    p.R1 = R1;
    p.nslice = nslice;
    fused_finish(p);
    return p;
}

// Makespan of a plan's work list on `sms` CTAs that each take the next ticket when free, in
// units of one SCAN sub-chunk: a STATE sub-chunk (the update MMA and w o x only) costs about
// 0.45 of one, each item about 0.25 more (its first loads and last drain are only partly
// hidden), a PASS item 0.3 plus 0.02 per chained super-chunk; a PASS item starts after the
// STATE items of its pair end, a SCAN item of super-chunk m >= 1 after the PASS items of its
// pair end.
inline double fused_makespan(const FusedPlan &p, int sms)
{
    const double c_scan = 1.0, c_state = 0.45, c_item = 0.25, c_pass0 = 0.3, c_pass1 = 0.02;
    const int grid = std::min(sms, p.n_items);
    std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
    for (int i = 0; i < grid; ++i) free_at.push(0.0);
    std::vector<double> state_end(p.npair, 0.0), pass_end(p.npair, 0.0);
    double span = 0.0;
    for (int t = 0; t < p.n_items; ++t) {
        const FusedItem it = fused_item(p, t);
        double s = free_at.top();
        free_at.pop();
        double e;
        if (it.kind == kItemState) {
            e = s + c_item + it.nq * c_state;
            state_end[it.pair] = std::max(state_end[it.pair], e);
        } else if (it.kind == kItemPass) {
            s = std::max(s, state_end[it.pair]);
            e = s + c_pass0 + c_pass1 * (it.nsup - 1);
            pass_end[it.pair] = std::max(pass_end[it.pair], e);
        } else {
            if (it.m > 0) s = std::max(s, pass_end[it.pair]);
            e = s + c_item + it.nq * c_scan;
        }
        free_at.push(e);
        span = std::max(span, e);
    }
    return span;
}

// The plan with the shortest simulated makespan among: every sequence cut into nsup equal
// super-chunks (nsup = 1 .. nc), and whole sequences for all pairs but a tail of k pairs
// (k = npair - w * sms: the pairs of a last, partial wave) cut into nsup1 super-chunks.  At
// most nc super-chunks per sequence (the workspace holds one state per chunk) and 64.
inline FusedPlan fused_search(int npair, int nsub, int nc, int sms, int nslice)
{
    const int max_sup = std::min(nc, std::min(nsub, 64));
    FusedPlan best = fused_candidate(npair, nsub, npair, nsub, nsub, nslice);
    double best_t = fused_makespan(best, sms);
    auto consider = [&](const FusedPlan &p) {
        const double t = fused_makespan(p, sms);
        if (t < best_t * 0.999 || (t <= best_t * 1.001 && p.n_items < best.n_items)) { best = p; best_t = t; }
    };
    int last_R = nsub;
    for (int want = 2; want <= max_sup; ++want) {
        const int R = (nsub + want - 1) / want;
        if (R == last_R || (nsub + R - 1) / R > max_sup) continue;
        last_R = R;
        consider(fused_candidate(npair, nsub, npair, R, R, nslice));
    }
    for (int w = 1; w <= 3; ++w) {
        const int k = npair - w * sms;
        if (k <= 0 || k >= npair) break;
        int last1 = nsub;
        for (int want = 2; want <= max_sup; ++want) {
            const int R1 = (nsub + want - 1) / want;
            if (R1 == last1 || (nsub + R1 - 1) / R1 > max_sup) continue;
            last1 = R1;
            consider(fused_candidate(npair, nsub, npair - k, nsub, R1, nslice));
        }
    }
    return best;
}

}  // namespace ssd
