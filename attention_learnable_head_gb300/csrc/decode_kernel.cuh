// Decode forward of attention with a per-head sink over a paged key/value
// cache, sm_103a.
//
// One new query token per sequence attends every cached key of its sequence
// (the last row of the causal concat-sink attention: listing
// "带汇聚的注意力（GPT-OSS）" of the euno.news page with N_q = 1), or the last W
// keys with a window.  The cache is paged: k_cache / v_cache
// [num_pages, page_size, H_kv, 64] bf16, block_table[b, p] = page holding keys
// [p * page_size, (p + 1) * page_size) of sequence b.
//
// Split-KV: CTA (split, kv head g, sequence b) attends the G = H_q / H_kv
// query heads of g to one slice of b's keys, without the sink, and writes the
// slice's normalised result and log-sum-exp; attn_sink_merge_kernel then adds
// the sink once (the merge of the key-chunk forward).  The work is a skinny
// contraction (G <= 8 rows) meant to be bound by reading the cache: it runs on the
// CUDA cores in fp32.  Each key is handled by 8 lanes, each holding 8 of the 64
// dimensions (one 16-byte load of K and of V); the lanes of a key combine the
// G dot products with three shuffles, and every lane keeps its own online
// softmax state for its keys.  The 16 states of a CTA (4 warps x 4 keys in
// flight) are merged through shared memory at the end.
#pragma once
#include <cuda_bf16.h>
#include "sm103_ptx.cuh"

namespace attn_sink {

constexpr int kDecThreads = 128;
constexpr int kDecMaxGroup = 8;        // query heads per kv head
constexpr int kDecStates = kDecThreads / 8;   // key groups of 8 lanes per CTA
constexpr float kLn2Dec = 0.6931471805599453f;
constexpr int kDecUnroll = 2;       // keys per key group whose loads are in flight together

struct DecodeParams {
  const __nv_bfloat16* q;         // [B][H_q][64]
  const __nv_bfloat16* k_cache;   // [num_pages][page_size][H_kv][64]
  const __nv_bfloat16* v_cache;
  const int* block_table;         // [B][max_pages]
  const int* seq_lens;            // [B]
  __nv_bfloat16* o_part;          // [splits][B][H_q][64] slice results
  __nv_bfloat16* o_part_lo;       // residuals of o_part
  float* lse_part;                // [splits][H_q][B] (natural log), -inf: no key
  int* err;
  int batch, heads_q, heads_kv;
  int page_size, num_pages, max_pages;
  int window;
  int splits;
  float scale_log2;               // softmax_scale * log2(e)
};

// G = query heads per kv head (1, 2, 4 or 8), a compile-time constant so that
// the G independent score / softmax chains of a key are interleaved.
template <int G>
__global__ void __launch_bounds__(kDecThreads) attn_sink_decode_kernel(const DecodeParams p) {
  __shared__ float s_m[kDecStates][G];
  __shared__ float s_l[kDecStates][G];
  __shared__ float s_o[kDecStates][G][64];

  const int split = blockIdx.x;
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int tid = threadIdx.x;
  const int state = tid >> 3;                  // key group of 8 lanes (0..15)
  const int ds = tid & 7;                      // dimension slice: dims [8 ds, 8 ds + 8)

  // keys [lo, hi) of this sequence, then this split's slice of them
  int L = __ldg(p.seq_lens + b);
  const int cap = p.max_pages * p.page_size;
  if (L < 0 || L > cap) {
    if (tid == 0) atomicCAS(p.err, 0, DEVERR_DECODE_INPUT);
    L = max(0, min(L, cap));
  }
  const int lo = p.window > 0 ? max(0, L - p.window) : 0;
  const int per = (L - lo + p.splits - 1) / p.splits;
  const int k0 = lo + split * per;
  const int k1 = min(L, k0 + per);

  // the G query rows of kv head g, dims of this lane, pre-scaled to log2 units
  float qv[G][8];
  #pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(
        p.q + ((size_t)b * p.heads_q + g * G + h) * 64 + 8 * ds));
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    #pragma unroll
    for (int e = 0; e < 4; ++e) {
      qv[h][2 * e] = bf16_lo(ww[e]) * p.scale_log2;
      qv[h][2 * e + 1] = bf16_hi(ww[e]) * p.scale_log2;
    }
  }
  float m[G], l[G], o[G][8];
  #pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.0f;
    #pragma unroll
    for (int e = 0; e < 8; ++e) o[h][e] = 0.0f;
  }

  const size_t row_stride = (size_t)p.heads_kv * 64;     // one key of the cache
  // Each key group takes kDecUnroll keys per step and issues their loads before
  // using them.  The trip count is the same for every lane of the CTA (k0, k1
  // are), so the shuffles always run with the whole warp.  The softmax update is
  // branch-free: a lane whose key is past the slice, or whose page entry is out
  // of range, uses a score of -inf, which changes neither m, l nor o.
  for (int jb = k0; jb < k1; jb += kDecUnroll * kDecStates) {
    uint4 kw[kDecUnroll], vw[kDecUnroll];
    bool valid[kDecUnroll];
    #pragma unroll
    for (int u = 0; u < kDecUnroll; ++u) {
      const int j = jb + u * kDecStates + state;
      valid[u] = j < k1;
      kw[u] = make_uint4(0, 0, 0, 0);
      vw[u] = make_uint4(0, 0, 0, 0);
      if (valid[u]) {
        const int pg = __ldg(p.block_table + (size_t)b * p.max_pages + j / p.page_size);
        if (pg < 0 || pg >= p.num_pages) {                // bounds check of the table
          if (ds == 0) atomicCAS(p.err, 0, DEVERR_DECODE_INPUT);
          valid[u] = false;
        } else {
          const size_t off =
              ((size_t)pg * p.page_size + j % p.page_size) * row_stride + g * 64 + 8 * ds;
          kw[u] = __ldg(reinterpret_cast<const uint4*>(p.k_cache + off));
          vw[u] = __ldg(reinterpret_cast<const uint4*>(p.v_cache + off));
        }
      }
    }
    #pragma unroll
    for (int u = 0; u < kDecUnroll; ++u) {
      const uint32_t kk[4] = {kw[u].x, kw[u].y, kw[u].z, kw[u].w};
      const uint32_t vv[4] = {vw[u].x, vw[u].y, vw[u].z, vw[u].w};
      float kf[8], vf[8];
      #pragma unroll
      for (int e = 0; e < 4; ++e) {
        kf[2 * e] = bf16_lo(kk[e]);
        kf[2 * e + 1] = bf16_hi(kk[e]);
        vf[2 * e] = bf16_lo(vv[e]);
        vf[2 * e + 1] = bf16_hi(vv[e]);
      }
      float sc[G];
      #pragma unroll
      for (int h = 0; h < G; ++h) {
        float s0 = qv[h][0] * kf[0], s1 = qv[h][1] * kf[1];
        #pragma unroll
        for (int e = 2; e < 8; e += 2) {
          s0 = fmaf(qv[h][e], kf[e], s0);
          s1 = fmaf(qv[h][e + 1], kf[e + 1], s1);
        }
        sc[h] = s0 + s1;
      }
      // the key's 8 lanes are consecutive: xor 1, 2, 4 stays within them
      #pragma unroll
      for (int x = 1; x < 8; x <<= 1) {
        #pragma unroll
        for (int h = 0; h < G; ++h) sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], x);
      }
      #pragma unroll
      for (int h = 0; h < G; ++h) {
        const float sv = valid[u] ? sc[h] : -INFINITY;
        const float mn = fmaxf(m[h], sv);                 // online softmax, log2 units
        const float mb = (mn == -INFINITY) ? 0.0f : mn;
        const float alpha = ex2_approx(m[h] - mb);        // 0 while m is -inf
        const float pe = ex2_approx(sv - mb);             // 0 for an invalid key
        l[h] = fmaf(l[h], alpha, pe);
        #pragma unroll
        for (int e = 0; e < 8; ++e) o[h][e] = fmaf(pe, vf[e], o[h][e] * alpha);
        m[h] = mn;
      }
    }
  }

  // merge the 16 key-group states of the CTA
  #pragma unroll
  for (int h = 0; h < G; ++h) {
    if (ds == 0) {
      s_m[state][h] = m[h];
      s_l[state][h] = l[h];
    }
    #pragma unroll
    for (int e = 0; e < 8; ++e) s_o[state][h][8 * ds + e] = o[h][e];
  }
  __syncthreads();
  // thread t: head t / 16, dims 4 (t % 16) .. + 4
  const int h = tid >> 4;
  const int d0 = 4 * (tid & 15);
  if (h < G) {
    float mm = -INFINITY;
    for (int st = 0; st < kDecStates; ++st) mm = fmaxf(mm, s_m[st][h]);
    float ll = 0.0f, acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (mm > -INFINITY) {
      for (int st = 0; st < kDecStates; ++st) {
        if (s_m[st][h] == -INFINITY) continue;
        const float w = ex2_approx(s_m[st][h] - mm);
        ll = fmaf(w, s_l[st][h], ll);
        #pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = fmaf(w, s_o[st][h][d0 + e], acc[e]);
      }
    }
    const float inv = (ll > 0.0f) ? 1.0f / ll : 0.0f;
    const int hq = g * G + h;
    const size_t oi = (((size_t)split * p.batch + b) * p.heads_q + hq) * 64 + d0;
    uint32_t hi[2], lo2[2];
    #pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float f0 = acc[2 * e] * inv, f1 = acc[2 * e + 1] * inv;
      hi[e] = pack_bf16x2(f0, f1);
      lo2[e] = pack_bf16x2(f0 - bf16_lo(hi[e]), f1 - bf16_hi(hi[e]));
    }
    *reinterpret_cast<uint2*>(p.o_part + oi) = make_uint2(hi[0], hi[1]);
    *reinterpret_cast<uint2*>(p.o_part_lo + oi) = make_uint2(lo2[0], lo2[1]);
    if (d0 == 0)
      p.lse_part[((size_t)split * p.heads_q + hq) * p.batch + b] =
          (ll > 0.0f) ? (mm + __log2f(ll)) * kLn2Dec : -INFINITY;
  }
}

}  // namespace attn_sink
