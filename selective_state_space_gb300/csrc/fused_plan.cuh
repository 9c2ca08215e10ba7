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
// Items form four streams, each in a fixed internal order (super-chunk-major, pairs fastest,
// part 0 before part 1; the pairs of one B/C group are next to each other):
//   STATE  the states of super-chunks 0 .. nsup-2 of the cut pairs;
//   SCAN0  the SCAN items of super-chunk 0 of every pair (whole sequences included);
//   PASS   the PASS items (slice-major);
//   SCAN1  the SCAN items of super-chunks >= 1.
// The ticket order is a list of runs, each taking the next items of one stream:
// [SCAN0 x k0 | STATE | PASS | SCAN0 rest | SCAN1] (empty runs dropped), k0 chosen by the
// planner.  A PASS item waits for every STATE item of its pair, a SCAN item of super-chunk
// m >= 1 for every PASS item of its pair; both wait only on items of lower tickets, which
// running CTAs have already taken, so the waits always end.
constexpr int kFusedMaxRuns = 5;
enum FusedStream { kStreamState = 0, kStreamScan0 = 1, kStreamPass = 2, kStreamScan1 = 3 };

struct FusedPlan {
    int npair;            // two-head pairs (B * nh / 2)
    int nsub;             // 128-token sub-chunks per sequence
    int split;            // pairs of part 0
    int R0, nsup0;        // part 0: sub-chunks per super-chunk, super-chunks per sequence
    int R1, nsup1;        // part 1
    int nslice;           // PASS slices per cut pair
    int n_state0, n_state1, n_pass, n_scan0, n_scan1, n_items;   // n_scan*: SCAN items per part
    long long sbase1;     // state slot of part 1's first sequence
    int nrun;             // runs of the ticket order: stream, first ticket, first index in the stream
    int run_stream[kFusedMaxRuns], run_ticket[kFusedMaxRuns], run_first[kFusedMaxRuns];
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

// The ticket order [SCAN0 x k0 | STATE | PASS | SCAN0 rest | SCAN1] of a plan whose counts are
// set (0 <= k0 <= npair; empty runs are dropped).
__host__ __device__ inline void fused_order(FusedPlan &p, int k0)
{
    const int n_state = p.n_state0 + p.n_state1, n_scan1 = p.n_scan0 + p.n_scan1 - p.npair;
    const int streams[5] = {kStreamScan0, kStreamState, kStreamPass, kStreamScan0, kStreamScan1};
    const int counts[5] = {k0, n_state, p.n_pass, p.npair - k0, n_scan1};
    const int firsts[5] = {0, 0, 0, k0, 0};
    p.nrun = 0;
    int t = 0;
    for (int i = 0; i < 5; ++i) {
        if (counts[i] <= 0) continue;
        p.run_stream[p.nrun] = streams[i];
        p.run_ticket[p.nrun] = t;
        p.run_first[p.nrun] = firsts[i];
        ++p.nrun;
        t += counts[i];
    }
}

// Fill the item counts of a plan whose cut (npair, nsub, split, R0, R1, nslice) is set; the
// order starts as k0 = 0.
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
    fused_order(p, 0);
}

__host__ __device__ inline FusedItem fused_item(const FusedPlan &p, int t)
{
    int run = 0;
    while (run + 1 < p.nrun && t >= p.run_ticket[run + 1]) ++run;
    const int stream = p.run_stream[run], i = p.run_first[run] + (t - p.run_ticket[run]);
    FusedItem it;
    it.slice = 0;
    int part1;
    const int np0 = p.split, np1 = p.npair - p.split;
    if (stream == kStreamState) {
        it.kind = kItemState;
        part1 = i >= p.n_state0;
        const int j = part1 ? i - p.n_state0 : i;
        const int np = part1 ? np1 : np0;
        it.m = j / np;
        it.pair = (part1 ? p.split : 0) + j % np;
    } else if (stream == kStreamScan0) {
        it.kind = kItemScan;
        part1 = i >= np0;
        it.m = 0;
        it.pair = i;
    } else if (stream == kStreamPass) {
        it.kind = kItemPass;
        const int ncut0 = fused_cut0(p), ncut = ncut0 + fused_cut1(p);
        it.slice = i / ncut;
        const int c = i % ncut;
        part1 = c >= ncut0;
        it.pair = part1 ? p.split + (c - ncut0) : c;
        it.m = 0;
    } else {
        it.kind = kItemScan;
        const int rest0 = p.n_scan0 - np0;                // SCAN items of super-chunks >= 1, part 0
        part1 = i >= rest0;
        const int j = part1 ? i - rest0 : i;
        const int np = part1 ? np1 : np0;
        it.m = 1 + j / np;
        it.pair = (part1 ? p.split : 0) + j % np;
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
// units of one SCAN sub-chunk (about 2.8 us on GB300 for two heads).  Calibrated from per-item
// timestamps: an item costs about one unit more than its sub-chunks (its first loads, the
// entering state and the last drain are only partly hidden), a STATE sub-chunk about 0.6 of a
// SCAN one (the update MMA and w o x only, but x and B still come from HBM), a PASS item about
// 1.3 units plus 0.02 per chained super-chunk (a bulk-copy round trip, the stores and a
// fence), and the first item of each CTA one unit more (the CTA's own start).  A PASS item
// starts after the STATE items of its pair end, a SCAN item of super-chunk m >= 1 after the
// PASS items of its pair end.
inline double fused_makespan(const FusedPlan &p, int sms)
{
    const double c_scan = 1.0, c_state = 0.6, c_item = 1.0, c_pass0 = 1.3, c_pass1 = 0.02, c_start = 1.0;
    const int grid = std::min(sms, p.n_items);
    std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
    for (int i = 0; i < grid; ++i) free_at.push(c_start);
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
// super-chunks (nsup = 1 .. 64), and whole sequences for all pairs but a tail of k pairs
// (k = npair - w * sms: the pairs of a last, partial wave) cut into nsup1 super-chunks; each
// with k0 = 0, npair / 8, npair / 4, npair / 2 or npair SCAN items of super-chunk 0 ahead of the
// STATE items.  The state slots of all cut sequences together (two per pair and super-chunk)
// must fit the workspace's `slots`.
inline FusedPlan fused_search(int npair, int nsub, long long slots, int sms, int nslice)
{
    const int max_sup = std::min(nsub, 64);
    FusedPlan best = fused_candidate(npair, nsub, npair, nsub, nsub, nslice);
    double best_t = fused_makespan(best, sms);
    auto consider = [&](FusedPlan p) {
        const long long used = 2LL * fused_cut0(p) * p.nsup0 + 2LL * fused_cut1(p) * p.nsup1;
        if (used > slots) return;
        const int k0s[5] = {0, npair / 8, npair / 4, npair / 2, npair};
        for (int i = 0; i < 5; ++i) {
            if (i > 0 && k0s[i] == k0s[i - 1]) continue;
            fused_order(p, k0s[i]);
            const double t = fused_makespan(p, sms);
            if (t < best_t * 0.999 || (t <= best_t * 1.001 && p.n_items < best.n_items)) {
                best = p;
                best_t = t;
            }
        }
    };
    int last_R = nsub;
    for (int want = 2; want <= max_sup; ++want) {
        const int R = (nsub + want - 1) / want;
        if (R == last_R) continue;
        last_R = R;
        consider(fused_candidate(npair, nsub, npair, R, R, nslice));
    }
    for (int w = 1; w <= 3; ++w) {
        const int k = npair - w * sms;
        if (k <= 0 || k >= npair) break;
        int last1 = nsub;
        for (int want = 2; want <= max_sup; ++want) {
            const int R1 = (nsub + want - 1) / want;
            if (R1 == last1) continue;
            last1 = R1;
            consider(fused_candidate(npair, nsub, npair - k, nsub, R1, nslice));
        }
    }
    return best;
}

}  // namespace ssd
