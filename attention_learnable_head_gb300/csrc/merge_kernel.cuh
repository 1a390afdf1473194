// Sink-aware merge of attention results over key chunks, sm_103a.
//
// Each chunk c gave, for query row i of head h, O_c (attention over the
// chunk's keys alone, normalised within the chunk; bf16 plus an optional bf16
// residual) and LSE_c = log sum_{j in c} exp(S_ij) (-inf when the row saw no
// key of the chunk).  Over the widened row [S_chunk_1 | ... | S_chunk_C | sink]
// of the concat listing "带汇聚的注意力（GPT-OSS）" (euno.news page), with
// Z = sum_c exp(LSE_c) + exp(sink[h]):
//   O = sum_c exp(LSE_c - log Z) O_c,   LSE = log Z,
// so the sink enters the normaliser once.  HBM-bound: eight threads per
// (row, head), each owning 8 of the 64 output columns (one 16-byte load per
// chunk and per tensor).
#pragma once
#include <cuda_bf16.h>
#include "sm103_ptx.cuh"

namespace attn_sink {

struct MergeParams {
  const __nv_bfloat16* o_parts;    // [C][T][H][64]
  const __nv_bfloat16* res_parts;  // [C][T][H][64] residuals, or null
  const float* lse_parts;          // [C][H][T]
  const float* sink;               // [H]
  __nv_bfloat16* out;              // [T][H][64]
  __nv_bfloat16* out_lo;           // [T][H][64] residual of out, or null
  float* lse;                      // [H][T]
  int num_chunks, total_q, heads_q;
};

__global__ void __launch_bounds__(256) attn_sink_merge_kernel(const MergeParams p) {
  const size_t pairs = (size_t)p.total_q * p.heads_q;
  const size_t stride = (size_t)gridDim.x * (blockDim.x >> 3);
  const int sub = threadIdx.x & 7;                    // 16-byte slice of the 128-byte row
  for (size_t pr = (size_t)blockIdx.x * (blockDim.x >> 3) + (threadIdx.x >> 3); pr < pairs;
       pr += stride) {
    const int t = (int)(pr / p.heads_q);
    const int h = (int)(pr % p.heads_q);
    const size_t lse_idx = (size_t)h * p.total_q + t;
    const size_t chunk_lse = (size_t)p.heads_q * p.total_q;
    const size_t chunk_o = (size_t)p.total_q * p.heads_q * 64;
    // m = max over the chunks' LSE and the sink (natural log)
    const float s = __ldg(p.sink + h);
    float m = s;
    for (int c = 0; c < p.num_chunks; ++c) m = fmaxf(m, __ldg(p.lse_parts + c * chunk_lse + lse_idx));
    const float m_use = (m == -INFINITY) ? 0.0f : m;
    float z = (s == -INFINITY) ? 0.0f : __expf(s - m_use);
    float acc[8];
    #pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
    const size_t o_idx = pr * 64 + sub * 8;
    for (int c = 0; c < p.num_chunks; ++c) {
      const float lc = __ldg(p.lse_parts + c * chunk_lse + lse_idx);
      if (lc == -INFINITY) continue;                  // the row saw no key of chunk c
      const float w = __expf(lc - m_use);
      z += w;
      const uint4 o = __ldg(reinterpret_cast<const uint4*>(p.o_parts + c * chunk_o + o_idx));
      const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
      uint32_t rw[4] = {0u, 0u, 0u, 0u};
      if (p.res_parts) {
        const uint4 r = __ldg(reinterpret_cast<const uint4*>(p.res_parts + c * chunk_o + o_idx));
        rw[0] = r.x; rw[1] = r.y; rw[2] = r.z; rw[3] = r.w;
      }
      #pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc[2 * u] = fmaf(w, bf16_lo(ow[u]) + bf16_lo(rw[u]), acc[2 * u]);
        acc[2 * u + 1] = fmaf(w, bf16_hi(ow[u]) + bf16_hi(rw[u]), acc[2 * u + 1]);
      }
    }
    const float inv_z = (z > 0.0f) ? 1.0f / z : 0.0f;
    uint32_t hi[4], lo[4];
    #pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float f0 = acc[2 * u] * inv_z, f1 = acc[2 * u + 1] * inv_z;
      hi[u] = pack_bf16x2(f0, f1);
      lo[u] = pack_bf16x2(f0 - bf16_lo(hi[u]), f1 - bf16_hi(hi[u]));
    }
    *reinterpret_cast<uint4*>(p.out + o_idx) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    if (p.out_lo)
      *reinterpret_cast<uint4*>(p.out_lo + o_idx) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    if (sub == 0) p.lse[lse_idx] = (z > 0.0f) ? m_use + __logf(z) : -INFINITY;
  }
}

}  // namespace attn_sink
