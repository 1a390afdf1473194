// Work order for packed batches of several sequences: every 128-row tile of
// every sequence (query tiles for the forward, key tiles for the backward),
// sorted by its cost (the number of tiles on the other side it meets under the
// mask), longest first.  The forward and backward grids then index this table
// instead of a dense (tile, sequence) grid: no CTA is launched for a tile past
// its sequence's end, and the heaviest tiles of all sequences start first, so
// the last CTAs to run are short ones.
//
// One CTA of 1024 threads: a counting sort over the costs (clamped to the
// histogram's size; ties in any order, which changes no result, since each
// tile's outputs are its own).  Entries are seq << 16 | tile; slots past the
// number of tiles hold kNoWork.
#pragma once
#include "fwd_kernel.cuh"

namespace attn_sink {

constexpr int kSchedThreads = 1024;
constexpr int kSchedBuckets = 2048;     // costs >= this share the top bucket

struct SchedParams {
  const int* cu_q;
  const int* cu_k;
  int num_seqs;
  int causal, window;
  int chunk, q_pos0;   // forward key-chunk mode (query row i at key i + q_pos0)
  int by_keys;         // 0: query tiles (forward), 1: key tiles (backward)
  int n_slots;         // table entries (>= the number of tiles)
  uint32_t* table;
};

// Tiles of sequence s on the sorted side, and the cost of tile t.
__device__ __forceinline__ int sched_tiles(const SchedParams& p, const SeqSpan& sp) {
  const int n = p.by_keys ? sp.nk : sp.nq;
  return (n + kBlockM - 1) / kBlockM;
}

__device__ __forceinline__ int sched_cost(const SchedParams& p, const SeqSpan& sp, int t) {
  if (!p.by_keys) {
    // key tiles a query tile meets (as the forward computes them)
    const int r0 = t * kBlockM;
    const int r1 = min(r0 + kBlockM, sp.nq) - 1;
    const int off = p.chunk ? p.q_pos0 : sp.nk - sp.nq;
    return key_tiles(r0, r1, sp, off, p.causal, p.window).num;
  }
  // query tiles a key tile meets (as the backward computes them)
  const int j0 = t * kBlockN;
  const int last_key = min(j0 + kBlockN, sp.nk) - 1;
  const int off = sp.nk - sp.nq;
  int q_lo = 0, q_hi = sp.nq;
  if (p.causal) {
    q_lo = max(0, j0 - off);
    if (p.window > 0) q_hi = min(sp.nq, last_key - off + p.window);
  }
  return (q_hi > q_lo) ? ((q_hi + kBlockM - 1) / kBlockM - q_lo / kBlockM) : 0;
}

__global__ void __launch_bounds__(kSchedThreads, 1)
attn_sink_schedule_kernel(const SchedParams p) {
  __shared__ int hist[kSchedBuckets];
  __shared__ int warp_sums[kSchedThreads / 32];
  const int tid = threadIdx.x;
  for (int b = tid; b < kSchedBuckets; b += kSchedThreads) hist[b] = 0;
  for (int i = tid; i < p.n_slots; i += kSchedThreads) p.table[i] = kNoWork;
  __syncthreads();
  // histogram of costs, bucket = (kSchedBuckets - 1) - min(cost, top): the
  // heaviest tiles get the lowest slots
  for (int s = tid; s < p.num_seqs; s += kSchedThreads) {
    const SeqSpan sp = seq_span(p.cu_q, p.cu_k, s, 0, 0);
    const int nt = sched_tiles(p, sp);
    for (int t = 0; t < nt; ++t) {
      const int c = min(sched_cost(p, sp, t), kSchedBuckets - 1);
      atomicAdd(&hist[kSchedBuckets - 1 - c], 1);
    }
  }
  __syncthreads();
  // exclusive prefix sum over the buckets: each thread owns 2 consecutive buckets
  constexpr int kPer = kSchedBuckets / kSchedThreads;
  int local[kPer];
  int run = 0;
  #pragma unroll
  for (int u = 0; u < kPer; ++u) {
    local[u] = hist[tid * kPer + u];
    run += local[u];
  }
  const int lane = tid & 31, warp = tid >> 5;
  int incl = run;
  #pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
    #pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;   // inclusive over warps
  }
  __syncthreads();
  int base = incl - run + (warp > 0 ? warp_sums[warp - 1] : 0);
  #pragma unroll
  for (int u = 0; u < kPer; ++u) {
    hist[tid * kPer + u] = base;    // first slot of the bucket
    base += local[u];
  }
  __syncthreads();
  // scatter
  for (int s = tid; s < p.num_seqs; s += kSchedThreads) {
    const SeqSpan sp = seq_span(p.cu_q, p.cu_k, s, 0, 0);
    const int nt = sched_tiles(p, sp);
    for (int t = 0; t < nt; ++t) {
      const int c = min(sched_cost(p, sp, t), kSchedBuckets - 1);
      const int pos = atomicAdd(&hist[kSchedBuckets - 1 - c], 1);
      if (pos < p.n_slots) p.table[pos] = ((uint32_t)s << 16) | (uint32_t)t;
    }
  }
}

}  // namespace attn_sink
