// Work split of the indexer scoring kernels (bf16 and MXFP4): a persistent
// grid of at most one CTA per SM walks "jobs", each a (query group, chunk of
// 128-entry tiles) pair.  Tiles past a group's causal limit are never loaded.
#pragma once
#include "common.cuh"

namespace sa {

constexpr int kTileEntries = 128;     // cache entries per tile (the MMA M)
constexpr int kIdxHeads = 64;         // indexer heads (the MMA N per query)
constexpr int kIdxDim = 64;           // indexer key width (the MMA K)
constexpr int kMaxJobsPerCta = 256;   // job table entries in shared memory

template <int QG>
struct JobRec {
  int b, t0, nq, t_lo, t_hi, g;
  int n[QG];            // visible entries of each query of the group
};

struct ScoreJobs {
  const float* w;       // [B*T, 64] head weights
  const int32_t* q_pos;
  int B, T, m, N_cap;
  int chunk_tiles, max_chunks;
  int64_t njobs;
  int contiguous;       // 1: each CTA takes one contiguous run of jobs
  float* scores;
  int64_t ld;
  int32_t* err;
};

template <int QG>
__device__ __forceinline__ JobRec<QG> make_job(const ScoreJobs& p, int64_t job) {
  JobRec<QG> J;
  const int64_t g = job / p.max_chunks;
  const int c = (int)(job % p.max_chunks);
  const int gpb = (p.T + QG - 1) / QG;
  J.g = (int)g;
  J.b = (int)(g / gpb);
  J.t0 = (int)(g % gpb) * QG;
  J.nq = min(QG, p.T - J.t0);
  int64_t nmax = 0;
#pragma unroll
  for (int q = 0; q < QG; ++q) {
    int64_t n = 0;
    if (q < J.nq) {
      const int pos = __ldg(p.q_pos + (int64_t)J.b * p.T + J.t0 + q);
      n = pos < 0 ? 0 : min64(((int64_t)pos + 1) / p.m, p.N_cap);
    }
    J.n[q] = (int)n;
    nmax = max64(nmax, n);
  }
  const int ntiles = (int)((nmax + kTileEntries - 1) / kTileEntries);
  J.t_lo = c * p.chunk_tiles;
  J.t_hi = min(ntiles, J.t_lo + p.chunk_tiles);
  return J;
}

// Fill this CTA's job table.  Contiguous order: CTA c takes jobs
// [c*J/G, (c+1)*J/G), so its tiles run along one or two query groups and the
// query tile is rarely reloaded.  Strided order: CTA c takes jobs c, c+G, ...,
// which balances groups of very different causal lengths (prefill).
// Returns the number of jobs of this CTA.
template <int QG>
__device__ __forceinline__ int fill_job_table(const ScoreJobs& p, JobRec<QG>* jobs) {
  int n_my;
  int64_t j_first, j_step;
  if (p.contiguous) {
    const int64_t lo = p.njobs * blockIdx.x / gridDim.x;
    const int64_t hi = p.njobs * (blockIdx.x + 1) / gridDim.x;
    n_my = (int)(hi - lo);
    j_first = lo;
    j_step = 1;
  } else {
    n_my = (int)((p.njobs - blockIdx.x + gridDim.x - 1) / gridDim.x);
    j_first = blockIdx.x;
    j_step = gridDim.x;
  }
  for (int i = threadIdx.x; i < n_my; i += blockDim.x)
    jobs[i] = make_job<QG>(p, j_first + (int64_t)i * j_step);
  return n_my;
}

// Host: choose the chunking (about 16 jobs per CTA, never more than the job
// table holds; chunks a multiple of `step_tiles` where the shape allows, for
// kernels that take that many tiles at a time) and the job order.  Returns the
// grid size, 0 if there is no work, or -1 if the shape cannot be split into
// the job table.
inline int plan_score_jobs(ScoreJobs& p, int QG, int num_sms, int step_tiles = 1) {
  const int64_t ngroups = (int64_t)p.B * ((p.T + QG - 1) / QG);
  const int ntiles_max = (p.N_cap + kTileEntries - 1) / kTileEntries;
  if (ngroups == 0 || ntiles_max == 0) return 0;
  int64_t ct = (ngroups * ntiles_max) / (16LL * num_sms);
  if (ct < 1) ct = 1;
  ct = (ct + step_tiles - 1) / step_tiles * step_tiles;
  if (ct > ntiles_max) ct = ntiles_max;
  while (ct < ntiles_max &&
         ngroups * ((ntiles_max + ct - 1) / ct) > (int64_t)kMaxJobsPerCta * num_sms)
    ct *= 2;
  if (ct > ntiles_max) ct = ntiles_max;
  if (ngroups * ((ntiles_max + ct - 1) / ct) > (int64_t)kMaxJobsPerCta * num_sms) return -1;
  p.chunk_tiles = (int)ct;
  p.max_chunks = (int)((ntiles_max + ct - 1) / ct);
  p.njobs = ngroups * p.max_chunks;
  // Few query groups (decode): every group spans many CTAs, all of equal
  // length, so contiguous runs keep the query tile resident.  Many groups
  // (prefill): strided order balances their causal lengths.
  p.contiguous = ngroups <= 4 * (int64_t)num_sms ? 1 : 0;
  return (int)min64(num_sms, p.njobs);
}

}  // namespace sa
