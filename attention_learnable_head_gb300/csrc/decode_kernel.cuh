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
// slice's normalised result and log-sum-exp.  The last of the (b, g) CTAs to
// finish (a counter per (b, g), zeroed before the launch) merges the slices
// and adds the sink once, as attn_sink_merge_kernel does for key chunks, so a
// decode step is one launch.
//
// The G query heads are the rows of a skinny product (G <= 8, padded to the 16
// rows of a warp-level mma.sync m16n8k16; a tcgen05 MMA needs 64 or more rows).
// Blocks of 64 keys of K and V are copied into swizzled shared memory with
// cp.async (two stages, page by page through the block table, rows past the
// slice or behind a bad table entry zero-filled and masked); each of the 4
// warps takes 16 keys of a block:
//   S = Q K^T   (bf16 operands: exact products, fp32 accumulators; K read with
//                ldmatrix as the column-major B operand)
//   online softmax per head row in fp32 (exp2 domain)
//   O += P V    (P and V as fp16, like the prefill forward's P V product; V
//                read with a transposing ldmatrix and converted from bf16)
// The 4 warps' (m, l, O) states are merged through shared memory at the end.
#pragma once
#include <cuda_bf16.h>
#include "sm103_ptx.cuh"

namespace attn_sink {

constexpr int kDecThreads = 128;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecMaxGroup = 8;        // query heads per kv head
constexpr int kDecKeys = 64;           // keys per stage: 16 per warp
constexpr int kDecStages = 2;
constexpr float kLn2Dec = 0.6931471805599453f;

struct DecodeParams {
  CUtensorMap tm_k;               // k_cache as [num_pages * page_size][H_kv][64], box
  CUtensorMap tm_v;               //   64 x 1 x min(page_size, 64), 128B swizzle (TMA path)
  const __nv_bfloat16* q;         // [B][H_q][64]
  const __nv_bfloat16* k_cache;   // [num_pages][page_size][H_kv][64]
  const __nv_bfloat16* v_cache;
  const int* block_table;         // [B][max_pages]
  const int* seq_lens;            // [B]
  __nv_bfloat16* o_part;          // [splits][B][H_q][64] slice results
  __nv_bfloat16* o_part_lo;       // residuals of o_part
  float* lse_part;                // [splits][H_q][B] (natural log), -inf: no key
  int* done;                      // [B][H_kv] CTAs of (b, g) finished (zero at launch)
  const float* sink;              // [H_q]
  __nv_bfloat16* out;             // [B][H_q][64]
  __nv_bfloat16* out_lo;          // residual of out, or null
  float* lse;                     // [H_q][B] (natural log)
  int* err;
  int batch, heads_q, heads_kv;
  int page_size, num_pages, max_pages;
  int window;
  int splits;
  int log2_page;                  // TMA path: log2(page_size)
  float scale_log2;               // softmax_scale * log2(e)
};

// Page sizes the TMA path copies whole: a multiple of 8 keys (whole 128-byte
// swizzle atoms) that divides the 64-key block or is a multiple of it.
__host__ __device__ constexpr bool decode_tma_page(int page_size) {
  return page_size >= 8 && (page_size & (page_size - 1)) == 0;
}

// G = query heads per kv head (1, 2, 4 or 8).  kTma: the blocks' pages are
// copied by TMA (one thread issues them; page sizes of decode_tma_page),
// otherwise by every thread with 16-byte cp.async.
template <int G, bool kTma>
__global__ void __launch_bounds__(kDecThreads, 5)
attn_sink_decode_kernel(const __grid_constant__ DecodeParams p) {
  __shared__ __align__(1024) uint8_t s_kv[kDecStages][2][kDecKeys * 128];   // K, V blocks
  __shared__ uint8_t s_valid[kDecStages][kDecKeys];    // key inside the slice, page in range
  __shared__ uint8_t s_pageok[kDecStages][8];          // TMA path: copy i of the block is a page
  __shared__ __align__(8) uint64_t kv_full[kDecStages];   // TMA path: the stage's copies landed
  __shared__ float s_m[kDecWarps][kDecMaxGroup];
  __shared__ float s_l[kDecWarps][kDecMaxGroup];
  __shared__ int s_last;
  // the warps' O rows for the final merge reuse the K/V stages (free by then)
  float (*s_o)[kDecMaxGroup][64] = reinterpret_cast<float (*)[kDecMaxGroup][64]>(&s_kv[0][0][0]);
  static_assert(sizeof(float) * kDecWarps * kDecMaxGroup * 64 <= sizeof(s_kv),
                "merge buffer larger than the K/V stages");

  const int split = blockIdx.x;
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int gr = lane >> 2;          // fragment row = query head of the group
  const int t4 = lane & 3;           // fragment column pair

  // keys [lo, hi) of this sequence, then this split's slice of them
  int L = __ldg(p.seq_lens + b);
  const int cap = p.max_pages * p.page_size;
  if (L < 0 || L > cap) {
    if (tid == 0) atomicCAS(p.err, 0, DEVERR_DECODE_INPUT);
    L = max(0, min(L, cap));
  }
  // The slices start on 64-key block boundaries (so the TMA path copies whole
  // pages into a block); keys before the window start are masked.
  const int lo = p.window > 0 ? max(0, L - p.window) : 0;
  const int lo_blk = lo & ~(kDecKeys - 1);
  const int per = ((L - lo_blk + p.splits - 1) / p.splits + kDecKeys - 1) & ~(kDecKeys - 1);
  const int k0 = lo_blk + split * per;
  const int k1 = min(L, k0 + per);
  const int nblk = k1 > k0 ? (k1 - k0 + kDecKeys - 1) / kDecKeys : 0;
  const size_t row_stride = (size_t)p.heads_kv * 64;     // one key of the cache

  // Q as the A operand (rows >= G are zero): a0 = dims 16 kk + 2 t4 .. + 1,
  // a2 = the same + 8, of head row gr; a1 = a3 = 0 (rows 8..15).
  uint32_t qa0[4], qa2[4];
  #pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    qa0[kk] = 0u;
    qa2[kk] = 0u;
    if (gr < G) {
      const uint32_t* qp = reinterpret_cast<const uint32_t*>(
          p.q + ((size_t)b * p.heads_q + g * G + gr) * 64 + 16 * kk + 2 * t4);
      qa0[kk] = __ldg(qp);
      qa2[kk] = __ldg(qp + 4);
    }
  }

  // Each thread copies 8 of a block's 16-byte chunks: K and V of the keys
  // kq(u) = (tid / 8 + 16 u) % 64, u = 0..3, chunk tid % 8.  The block-table
  // entries of its keys are read one block ahead (pages of block blk + 2 while
  // block blk + 1 is copied), so the copies never wait on a table lookup.
  auto fetch_pages = [&](int blk, int* pg) {
    #pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = k0 + blk * kDecKeys + (((tid >> 3) + 16 * u) & (kDecKeys - 1));
      pg[u] = (blk < nblk && j < k1)
                  ? __ldg(p.block_table + (size_t)b * p.max_pages + j / p.page_size)
                  : -1;
    }
  };
  // Block `blk` of the slice into stage `st`, with the table entries pg of its
  // keys.  A key past the slice, or whose table entry is out of range
  // (reported, nothing read), is zero-filled and marked invalid.
  auto load_block = [&](int blk, int st, const int* pg) {
    const int base = k0 + blk * kDecKeys;
    const int c = tid & 7;
    #pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int key = ((tid >> 3) + 16 * u) & (kDecKeys - 1);
      const int j = base + key;
      const bool inside = j >= lo && j < k1;
      const bool valid = inside && pg[u] >= 0 && pg[u] < p.num_pages;
      if (inside && !valid && c == 0) atomicCAS(p.err, 0, DEVERR_DECODE_INPUT);
      if (c == 0) s_valid[st][key] = valid ? 1 : 0;
      const size_t off = valid ? ((size_t)pg[u] * p.page_size + j % p.page_size) * row_stride +
                                     g * 64 + 8 * c
                               : 0;
      // with 0 bytes nothing is read: q is any valid address
      const __nv_bfloat16* ksrc = valid ? p.k_cache + off : p.q;
      const __nv_bfloat16* vsrc = valid ? p.v_cache + off : p.q;
      cp_async_16_zfill(smem_u32(&s_kv[st][0][0]) + sw128_offset(key, c), ksrc, valid ? 16 : 0);
      cp_async_16_zfill(smem_u32(&s_kv[st][1][0]) + sw128_offset(key, c), vsrc, valid ? 16 : 0);
    }
    cp_async_commit();
  };

  float m_r = -INFINITY;   // running max of head row gr (log2 units)
  float l_r = 0.0f;        // this thread's share of the row sum
  float oacc[8][4];        // O: n-tile nd = dims 8 nd .. 8 nd + 7 (c0, c1: row gr)
  #pragma unroll
  for (int nd = 0; nd < 8; ++nd) {
    #pragma unroll
    for (int e = 0; e < 4; ++e) oacc[nd][e] = 0.0f;
  }
  uint32_t vmag = 0;    // largest fp16 magnitude pattern of the converted V halves
  const int mi = lane >> 3, ri = lane & 7;   // ldmatrix: matrix and row this lane addresses
  const int kb = 16 * warp;                  // this warp's keys within a block

  // TMA path: thread 0 copies the pages of a block (boxes of min(page, 64)
  // keys; a page outside the cache is read at a coordinate beyond the tensor,
  // which fills zeros, and marked as such) and reads the block's table entries
  // one block ahead.  The consumers mask keys outside [lo, k1) and keys of a
  // page marked absent.
  const int log2_box = kTma ? min(p.log2_page, 6) : 0;
  const int box = 1 << log2_box;
  const int npg = kTma ? kDecKeys >> log2_box : 0;      // copies per block and tensor
  auto tma_fetch = [&](int blk, int* pe) {
    #pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int j = k0 + blk * kDecKeys + i * box;       // first key of copy i
      pe[i] = (i < npg && blk < nblk && j < k1)
                  ? __ldg(p.block_table + (size_t)b * p.max_pages + (j >> p.log2_page))
                  : -1;
    }
  };
  auto tma_issue = [&](int blk, int st, const int* pe) {
    const int base = k0 + blk * kDecKeys;
    const int oob = p.num_pages * p.page_size;           // first row past the cache
    int row[8];
    #pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int j = base + i * box;
      const bool needed = i < npg && j < k1 && j + box > lo;
      const bool ok = pe[i] >= 0 && pe[i] < p.num_pages;
      if (needed && !ok) atomicCAS(p.err, 0, DEVERR_DECODE_INPUT);
      row[i] = ok ? pe[i] * p.page_size + (j & (p.page_size - 1)) : oob;
      if (i < npg) s_pageok[st][i] = ok ? 1 : 0;
    }
    mbar_arrive_expect_tx(&kv_full[st], 2 * kDecKeys * 128);
    #pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < npg) {
        tma_load_3d(&p.tm_k, &kv_full[st], &s_kv[st][0][i * box * 128], 0, g, row[i]);
        tma_load_3d(&p.tm_v, &kv_full[st], &s_kv[st][1][i * box * 128], 0, g, row[i]);
      }
    }
  };
  int issued = 0;                                         // TMA path: blocks issued
  if (kTma) {
    if (tid == 0) {
      for (int st = 0; st < kDecStages; ++st) mbar_init(&kv_full[st], 1);
      fence_mbarrier_init();
    }
    __syncthreads();
  }

  // two-stage ring: block blk + 1 is in flight while blk is used (five CTAs per
  // SM keep ten blocks in flight; measured better than three stages at four
  // CTAs per SM)
  int pg[8], pg_next[8];
  bool ok = true;
  if (kTma) {
    if (tid == 0) {
      tma_fetch(0, pg);
      if (nblk > 0) tma_issue(0, 0, pg);
      tma_fetch(1, pg);
      if (nblk > 1) tma_issue(1, 1, pg);
      issued = min(nblk, 2);
      tma_fetch(2, pg_next);
    }
  } else {
    fetch_pages(0, pg);
    if (nblk > 0) load_block(0, 0, pg);
    fetch_pages(1, pg_next);
  }
  for (int blk = 0; blk < nblk; ++blk) {
    const int st = blk % kDecStages;
    if (kTma) {
      // bounded wait; the whole CTA agrees on the outcome
      const bool landed = mbar_wait_warp(&kv_full[st], (blk / kDecStages) & 1, nullptr);
      if (!__syncthreads_and(landed)) {
        ok = false;
        break;
      }
    } else {
      if (blk + 1 < nblk) {
        #pragma unroll
        for (int u = 0; u < 4; ++u) pg[u] = pg_next[u];
        fetch_pages(blk + 2, pg_next);
        load_block(blk + 1, (blk + 1) % kDecStages, pg);
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();
    }
    const uint32_t kt = smem_u32(&s_kv[st][0][0]);
    const uint32_t vt = smem_u32(&s_kv[st][1][0]);

    // S = Q K^T for keys kb .. kb + 15 (n-tiles of 8 keys); matrices of the x4
    // load: (keys +0, dims 16 kk), (keys +0, dims +8), (keys +8, ...), (keys +8, +8)
    float sc[2][4];
    #pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      #pragma unroll
      for (int e = 0; e < 4; ++e) sc[nt][e] = 0.0f;
    }
    #pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t b00, b01, b10, b11;
      ldmatrix_x4(kt + sw128_offset(kb + (mi >> 1) * 8 + ri, 2 * kk + (mi & 1)), b00, b01, b10,
                  b11);
      mma_16816_bf16(sc[0], qa0[kk], 0u, qa2[kk], 0u, b00, b01);
      mma_16816_bf16(sc[1], qa0[kk], 0u, qa2[kk], 0u, b10, b11);
    }

    // online softmax of row gr over keys kb + 8 nt + 2 t4 + e (log2 units)
    float x[2][2];
    float mx = -INFINITY;
    #pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      #pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = kb + 8 * nt + 2 * t4 + e;
        bool valid;
        if (kTma) {
          const int j = k0 + blk * kDecKeys + key;
          valid = s_pageok[st][key >> log2_box] != 0 && j >= lo && j < k1;
        } else {
          valid = s_valid[st][key] != 0;
        }
        x[nt][e] = valid ? sc[nt][e] * p.scale_log2 : -INFINITY;
        mx = fmaxf(mx, x[nt][e]);
      }
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mn = fmaxf(m_r, mx);
    const float mb = (mn == -INFINITY) ? 0.0f : mn;
    const float alpha = ex2_approx(m_r - mb);            // 0 while m is -inf
    float pv[2][2];
    float rs = 0.0f;
    #pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      #pragma unroll
      for (int e = 0; e < 2; ++e) {
        pv[nt][e] = ex2_approx(x[nt][e] - mb);           // 0 for an invalid key
        rs += pv[nt][e];
      }
    }
    l_r = fmaf(l_r, alpha, rs);
    m_r = mn;
    #pragma unroll
    for (int nd = 0; nd < 8; ++nd) {
      oacc[nd][0] *= alpha;
      oacc[nd][1] *= alpha;
    }
    // P as the A operand: a0 = keys 2 t4 .. + 1, a2 = keys 8 + 2 t4 .. + 1
    const uint32_t pa0 = pack_f16x2(pv[0][0], pv[0][1]);
    const uint32_t pa2 = pack_f16x2(pv[1][0], pv[1][1]);

    // O += P V; transposed x4 load matrices: (keys +0, dims 16 u), (keys +8,
    // dims 16 u), (keys +0, dims +8), (keys +8, dims +8)
    #pragma unroll
    for (int u = 0; u < 4; ++u) {
      uint32_t v0, v1, v2, v3;
      ldmatrix_x4_trans(vt + sw128_offset(kb + (mi & 1) * 8 + ri, 2 * u + (mi >> 1)), v0, v1,
                        v2, v3);
      const uint32_t h0 = bf16x2_to_f16x2_fast(v0), h1 = bf16x2_to_f16x2_fast(v1);
      const uint32_t h2 = bf16x2_to_f16x2_fast(v2), h3 = bf16x2_to_f16x2_fast(v3);
      vmag = __vmaxu2(vmag, __vmaxu2(h0 & 0x7fff7fffu, h1 & 0x7fff7fffu));
      vmag = __vmaxu2(vmag, __vmaxu2(h2 & 0x7fff7fffu, h3 & 0x7fff7fffu));
      mma_16816_f16(oacc[2 * u], pa0, 0u, pa2, 0u, h0, h1);
      mma_16816_f16(oacc[2 * u + 1], pa0, 0u, pa2, 0u, h2, h3);
    }
    __syncthreads();   // every warp is done with stage st before it is refilled
    if (kTma && tid == 0 && blk + 2 < nblk) {
      #pragma unroll
      for (int i = 0; i < 8; ++i) pg[i] = pg_next[i];
      tma_fetch(blk + 3, pg_next);
      tma_issue(blk + 2, st, pg);
      issued = blk + 3;
    }
  }
  if (!ok) {
    // a copy that did not land within the wait limit (the whole CTA agreed):
    // report it, give the copies still in flight (the last two issued) time to
    // land before the CTA releases its shared memory, and write nothing
    if (tid == 0) {
      atomicCAS(p.err, 0, DEVERR_TIMEOUT_FWD + 5);
      for (int j = max(0, issued - kDecStages); j < issued; ++j)
        mbar_wait(&kv_full[j % kDecStages], (j / kDecStages) & 1, nullptr);
    }
    return;
  }
  // a value that rounded to fp16 infinity (or a NaN) lies outside the fp16 range
  if ((vmag & 0xffffu) >= 0x7c00u || (vmag >> 16) >= 0x7c00u) atomicCAS(p.err, 0, DEVERR_FP16_RANGE);

  // the row sum over the 4 lanes of row gr, then the 4 warps' states merged
  l_r += __shfl_xor_sync(0xffffffffu, l_r, 1);
  l_r += __shfl_xor_sync(0xffffffffu, l_r, 2);
  if (gr < G) {
    if (t4 == 0) {
      s_m[warp][gr] = m_r;
      s_l[warp][gr] = l_r;
    }
    #pragma unroll
    for (int nd = 0; nd < 8; ++nd) {
      s_o[warp][gr][8 * nd + 2 * t4] = oacc[nd][0];
      s_o[warp][gr][8 * nd + 2 * t4 + 1] = oacc[nd][1];
    }
  }
  __syncthreads();
  // thread t: head t / 16, dims 4 (t % 16) .. + 4
  const int h = tid >> 4;
  const int d0 = 4 * (tid & 15);
  if (h < G) {
    float mm = -INFINITY;
    for (int w = 0; w < kDecWarps; ++w) mm = fmaxf(mm, s_m[w][h]);
    float ll = 0.0f, acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (mm > -INFINITY) {
      for (int w = 0; w < kDecWarps; ++w) {
        if (s_m[w][h] == -INFINITY) continue;
        const float wt = ex2_approx(s_m[w][h] - mm);
        ll = fmaf(wt, s_l[w][h], ll);
        #pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = fmaf(wt, s_o[w][h][d0 + e], acc[e]);
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

  // ---- the last CTA of (b, g) merges the slices with the sink:
  //   Z = sum_c exp(LSE_c) + exp(sink),  O = sum_c exp(LSE_c - log Z) O_c,
  //   LSE = log Z (natural log; the merge of the key-chunk forward).
  // Every CTA's slice results are visible before its count (fence, then the
  // atomic); the last one fences again before it reads the others'.
  __threadfence();
  __syncthreads();
  if (tid == 0)
    s_last = atomicAdd(p.done + (size_t)b * p.heads_kv + g, 1) == p.splits - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (h < G) {
    const int hq = g * G + h;
    const float sk = __ldg(p.sink + hq);
    float m = sk;
    for (int c = 0; c < p.splits; ++c)
      m = fmaxf(m, __ldcg(p.lse_part + ((size_t)c * p.heads_q + hq) * p.batch + b));
    const float m_use = (m == -INFINITY) ? 0.0f : m;
    float z = (sk == -INFINITY) ? 0.0f : __expf(sk - m_use);
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int c = 0; c < p.splits; ++c) {
      const float lc = __ldcg(p.lse_part + ((size_t)c * p.heads_q + hq) * p.batch + b);
      if (lc == -INFINITY) continue;                // the slice had no key
      const float wc = __expf(lc - m_use);
      z += wc;
      const size_t ci = (((size_t)c * p.batch + b) * p.heads_q + hq) * 64 + d0;
      const uint2 o = __ldcg(reinterpret_cast<const uint2*>(p.o_part + ci));
      const uint2 r = __ldcg(reinterpret_cast<const uint2*>(p.o_part_lo + ci));
      acc[0] = fmaf(wc, bf16_lo(o.x) + bf16_lo(r.x), acc[0]);
      acc[1] = fmaf(wc, bf16_hi(o.x) + bf16_hi(r.x), acc[1]);
      acc[2] = fmaf(wc, bf16_lo(o.y) + bf16_lo(r.y), acc[2]);
      acc[3] = fmaf(wc, bf16_hi(o.y) + bf16_hi(r.y), acc[3]);
    }
    const float inv_z = (z > 0.0f) ? 1.0f / z : 0.0f;
    uint32_t hi[2], lo2[2];
    #pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float f0 = acc[2 * e] * inv_z, f1 = acc[2 * e + 1] * inv_z;
      hi[e] = pack_bf16x2(f0, f1);
      lo2[e] = pack_bf16x2(f0 - bf16_lo(hi[e]), f1 - bf16_hi(hi[e]));
    }
    const size_t oi = ((size_t)b * p.heads_q + hq) * 64 + d0;
    *reinterpret_cast<uint2*>(p.out + oi) = make_uint2(hi[0], hi[1]);
    if (p.out_lo) *reinterpret_cast<uint2*>(p.out_lo + oi) = make_uint2(lo2[0], lo2[1]);
    if (d0 == 0) p.lse[(size_t)hq * p.batch + b] = (z > 0.0f) ? m_use + __logf(z) : -INFINITY;
  }
}

}  // namespace attn_sink
