// score_plan.cuh -- the work plan of the indexer scorer: query groups and the
// 128-pool tiles each one covers.  Built by one CTA: by every scorer CTA into
// its own shared memory (small batches), by the scorer's plan kernel, or by an
// extra CTA of the compression launch in the fused step.
#pragma once

#include "kp_common.cuh"

namespace kp {

constexpr int kScM = 128;   // pools per tile (MMA M)
constexpr int kScMaxQ = 8;  // queries per group

// Plan layout (int32 words) inside the score workspace.
struct PlanView {
    int32_t *hdr;      // [0] groups, [1] units, [2] queries in the largest group
    int32_t *q0;       // [NQ] first query of each group
    int32_t *nq;       // [NQ] queries in each group
    int32_t *seq;      // [NQ] sequence of each group
    int32_t *unit0;    // [NQ + 1] first unit of each group (exclusive scan of tiles)
    __host__ __device__ PlanView(int32_t *base, int n)
        : hdr(base), q0(base + 4), nq(base + 4 + n), seq(base + 4 + 2 * n), unit0(base + 4 + 3 * n) {}
};

// Groups runs of up to max_q (<= 8) adjacent queries of the same sequence and counts the
// 128-pool tiles each group needs (the largest n_full = (t + 1) >> kshift
// among its queries, 2^kshift tokens per pool).  A
// group whose sequence is out of range, or with a query at or past its
// sequence's length, gets no tiles and sets KP_ERR_DEVICE_BOUNDS.
// Every thread of the calling CTA must call it (blockDim.x a multiple of 32);
// `scratch` holds >= 33 ints of shared memory.
__device__ __forceinline__ void build_score_plan(int nq, int num_seqs, const int32_t *__restrict__ q_seq,
                                                 const int32_t *__restrict__ q_pos,
                                                 const int32_t *__restrict__ seq_len, int kshift, int max_tiles,
                                                 int32_t *plan_base, int32_t *status, int *scratch,
                                                 int max_q = kScMaxQ) {
    PlanView plan(plan_base, nq);
    int carry_run = -1, carry_groups = 0;
    for (int base = 0; base < nq; base += blockDim.x) {
        const int i = base + threadIdx.x;
        const bool in = i < nq;
        const int sq = in ? q_seq[i] : 0;
        const bool run_start = in && (i == 0 || q_seq[i - 1] != sq);
        int tot;
        int rs = block_inclusive_scan<1>(run_start ? i : -1, scratch, &tot);
        rs = max(rs, carry_run);
        carry_run = max(carry_run, tot);
        const bool gs = in && ((i - rs) % max_q == 0);
        const int incl = block_inclusive_scan<0>(gs ? 1 : 0, scratch, &tot);
        if (gs) {
            const int gid = carry_groups + incl - 1;
            plan.q0[gid] = i;
            plan.seq[gid] = sq;
        }
        carry_groups += tot;
    }
    __syncthreads();
    const int ng = carry_groups;
    int group_max = 0;
    for (int g = threadIdx.x; g < ng; g += blockDim.x) {
        const int q0 = plan.q0[g];
        const int q1 = (g + 1 < ng) ? plan.q0[g + 1] : nq;
        const int sq = plan.seq[g];
        const bool seq_ok = sq >= 0 && sq < num_seqs;
        const int len = seq_ok ? seq_len[sq] : 0;
        int mx = 0;
        bool pos_ok = true;
        for (int q = q0; q < q1; ++q) {
            const int t = q_pos[q];
            pos_ok = pos_ok && t < len;
            mx = max(mx, (t + 1) >> kshift);
        }
        int tiles = (mx + kScM - 1) / kScM;
        if (!seq_ok || !pos_ok) {
            set_status(status, KP_ERR_DEVICE_BOUNDS);
            tiles = 0;
        }
        if (tiles > max_tiles) {
            set_status(status, KP_ERR_DEVICE_BOUNDS);
            tiles = max_tiles;
        }
        plan.nq[g] = q1 - q0;
        plan.unit0[g] = tiles;
        group_max = max(group_max, q1 - q0);
    }
    __syncthreads();
    (void)block_inclusive_scan<1>(group_max, scratch, &group_max);
    int carry_units = 0;
    for (int base = 0; base < ng; base += blockDim.x) {
        const int g = base + threadIdx.x;
        const int v = g < ng ? plan.unit0[g] : 0;
        int tot;
        const int incl = block_inclusive_scan<0>(v, scratch, &tot);
        if (g < ng) plan.unit0[g] = carry_units + incl - v;
        carry_units += tot;
    }
    if (threadIdx.x == 0) {
        plan.unit0[ng] = carry_units;
        plan.hdr[0] = ng;
        plan.hdr[1] = carry_units;
        plan.hdr[2] = group_max;
    }
}

}  // namespace kp
