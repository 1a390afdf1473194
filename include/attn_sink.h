/*
 * attn_sink.h -- C ABI of libattn_sink.so: fused scaled-dot-product attention
 * with one learnable scalar sink logit per query head, forward and backward,
 * for NVIDIA GB300 (sm_103a).
 *
 * What is computed.  For query row i of head h (key/value head g = h / (H_q/H_kv)):
 *   S_ij = softmax_scale * <q_i, k_j>            over the keys j visible to i
 *   P_ij = exp(S_ij) / (sum_j' exp(S_ij') + exp(sink[h]))
 *   P_ih = exp(sink[h]) / (same denominator)
 *   out_i = sum_j P_ij v_j                          (the sink multiplies no value row)
 *   lse_i = log(sum_j exp(S_ij) + exp(sink[h]))      (natural log, sink included)
 * This is the concat-sink softmax of the listing "带汇聚的注意力（GPT-OSS）" and the
 * P_ij / P_ih equations (section "数学公式") on the page "解锁 GPT-OSS 的 Agentic RL
 * 训练：实用回顾" (euno.news); the same listing is on the page "Treinamento de RL
 * Agêntico para modelos GPT-OSS" (section "Desafio 3: Attention Sinks no
 * FlashAttention").  The sink is not multiplied by softmax_scale.
 *
 * Backward (section "反向传播" of the euno.news page for the sink; the ordinary
 * softmax-attention backward for the rest), with D_i = sum_d dout_i[d] * out_i[d]:
 *   dS_ij    = P_ij (<dout_i, v_j> - D_i)
 *   dq_i     = softmax_scale * sum_j dS_ij k_j
 *   dk_j     = softmax_scale * sum_{h in group, i} dS_ij q_i
 *   dv_j     = sum_{h in group, i} P_ij dout_i
 *   dsink[h] = - sum_i P_ih * D_i            (summed over every sequence)
 *
 * Masks.  causal: bottom-right aligned, query row i (0-based within its sequence)
 * sees key j iff j <= i + (N_k - N_q).  window W > 0 (requires causal): also
 * j > i + (N_k - N_q) - W, i.e. the W most recent keys including the diagonal.
 * A row that sees no key gets out = 0 and lse = sink[h].
 *
 * Layouts (all contiguous, head_dim innermost, token-major):
 *   q, out, dout, dq : [T_q, H_q, head_dim]     bf16 (dq: bf16 or fp32, see grad_dtype)
 *   k, v, dk, dv     : [T_k, H_kv, head_dim]    bf16 (dk, dv: bf16 or fp32)
 *   sink, dsink      : [H_q]                    fp32
 *   lse              : [H_q, T_q]               fp32
 *   cu_seqlens_q/k   : [num_seqs + 1]           int32, device memory, cu[0] = 0
 * Dense batches (cu_seqlens == NULL) use T_q = batch * seqlen_q, T_k = batch * seqlen_k,
 * sequence b occupying tokens [b*seqlen, (b+1)*seqlen).
 *
 * Ownership and threading.  Every pointer argument is DEVICE memory owned by the
 * caller (params is a host pointer read during the call only).  The library
 * allocates nothing.  Calls are asynchronous on `stream` (a cudaStream_t;
 * NULL = legacy default stream) and never synchronise the host.  All calls are
 * thread-safe; the global state is the cached driver entry point for
 * tensor-map encoding (initialised once), per-device launch attributes and a
 * launch counter.  Outputs are overwritten, never
 * accumulated into.  Device pointers of q, k, v, out, dout, dq, dk, dv must be
 * 16-byte aligned; the workspace must be 256-byte aligned.
 *
 * Errors.  Arguments are validated on the host before any launch; a bad
 * argument returns ATTN_SINK_ERR_INVALID_ARG / _UNSUPPORTED / _WORKSPACE and
 * launches nothing.  A failed launch returns ATTN_SINK_ERR_CUDA.  Every wait
 * inside the kernels is bounded: a wait that does not complete records an
 * error code in a device word (read it with attn_sink_device_error) and the
 * kernel returns instead of hanging.  The host never reads cu_seqlens.
 */
#ifndef ATTN_SINK_H
#define ATTN_SINK_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_SINK_OK = 0,
  ATTN_SINK_ERR_INVALID_ARG = 1,  /* null pointer, bad shape, misaligned pointer */
  ATTN_SINK_ERR_UNSUPPORTED = 2,  /* head_dim != 64, or a combination not built */
  ATTN_SINK_ERR_WORKSPACE = 3,    /* workspace missing or smaller than required */
  ATTN_SINK_ERR_CUDA = 4,         /* a CUDA runtime / driver call failed */
  ATTN_SINK_ERR_TIMEOUT = 5       /* a kernel gave up on a bounded wait */
} attn_sink_status;

/* Set the fields of one mode and leave the other mode's at 0: dense (batch,
 * seqlen_q, seqlen_k; cu_seqlens NULL) or packed (num_seqs, total_q, total_k,
 * max_seqlen_q, max_seqlen_k; cu_seqlens given).  Mixing them is an error. */
typedef struct attn_sink_params {
  /* dense batch (used when cu_seqlens_q == NULL) */
  int batch;
  int seqlen_q;
  int seqlen_k;
  /* packed variable-length sequences (used when cu_seqlens_q != NULL) */
  int num_seqs;
  int total_q;        /* T_q: tokens in q (= cu_seqlens_q[num_seqs]) */
  int total_k;        /* T_k */
  int max_seqlen_q;   /* upper bound on every query length; sizes the launch grid */
  int max_seqlen_k;   /* upper bound on every key length */
  /* heads */
  int heads_q;        /* H_q, a multiple of heads_kv */
  int heads_kv;       /* H_kv */
  int head_dim;       /* must be 64 */
  /* masking */
  int causal;         /* 0 or 1 */
  int window;         /* <= 0: no window; W > 0 needs causal = 1 */
  float softmax_scale;/* multiplies q.k only; finite and > 0 */
  /* backward outputs: 0 = bf16 dq/dk/dv, 1 = fp32 dq/dk/dv */
  int grad_dtype;
} attn_sink_params;

/*
 * Forward.  Writes out [T_q, H_q, 64] bf16 and lse [H_q, T_q] fp32.
 * out_residual (optional, NULL to skip): [T_q, H_q, 64] bf16, the rounding
 * residual of out (out + out_residual carries ~16 significand bits of O).
 * Passing it to attn_sink_bwd makes the backward's D_i = rowsum(dO o O) use
 * that O instead of the bf16 out, which matters where the softmax is peaked.
 * cu_seqlens_q and cu_seqlens_k are both NULL (dense) or both non-NULL (packed).
 * Arithmetic: S = q k^T on the bf16 inputs (exact products, fp32 sums); P and
 * v enter O = P v as fp16 (v is converted into the workspace first); O
 * accumulates in fp32.  v must lie within the fp16
 * range (|v| <= 65504), otherwise the device error word records
 * ATTN_SINK_DEVERR_FP16_RANGE (0x400).
 * Passage: listing "带汇聚的注意力（GPT-OSS）" and section "数学公式" of the
 * euno.news page.  Returns an attn_sink_status.
 */
int attn_sink_fwd(const attn_sink_params* params, const void* q, const void* k,
                  const void* v, const float* sink, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, void* out, void* out_residual, float* lse,
                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * Forward over one chunk of the keys, without the sink: for sequence
 * parallelism, where each piece of a long key sequence is attended separately
 * and the pieces are combined by attn_sink_merge.  Passage: the keryc.com page
 * on GPT-OSS agentic RL fixes, section "Solutions implemented by the team"
 * (sequence parallelism compatible with attention sinks), and the concat
 * listing "带汇聚的注意力（GPT-OSS）" of the euno.news page (the sink column
 * must enter the softmax once, so a chunk carries none).
 * k, v hold the chunk's keys (params->seqlen_k / cu_seqlens_k describe the
 * chunk).  q_pos0: key index within the chunk aligned with query row 0 of
 * every sequence: row i sees chunk key j iff j <= i + q_pos0 (causal) and
 * j > i + q_pos0 - W (window W > 0).  For the chunk that starts at key k0 of
 * a key sequence of length N_k queried by N_q rows, q_pos0 = N_k - N_q - k0;
 * |q_pos0| <= 2^30.  Ignored when params->causal = 0.
 * Writes out [T_q, H_q, 64] bf16 (attention over the chunk alone, normalised
 * within it), optional out_residual, and lse [H_q, T_q] = log sum_j exp(S_ij)
 * over the chunk (-inf, with out = 0, for rows that see no key of it).
 * Workspace, layouts, precision and errors as attn_sink_fwd; sink is not used.
 */
int attn_sink_fwd_chunk(const attn_sink_params* params, int q_pos0, const void* q,
                        const void* k, const void* v, const int* cu_seqlens_q,
                        const int* cu_seqlens_k, void* out, void* out_residual, float* lse,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * Sink-aware merge of num_chunks results of attn_sink_fwd_chunk over the
 * chunks of one key sequence:
 *   Z = sum_c exp(lse_c) + exp(sink[h]),  out = sum_c exp(lse_c - log Z) out_c,
 *   lse = log Z,
 * i.e. the attention of the whole key sequence with the sink counted once
 * (concat listing "带汇聚的注意力（GPT-OSS）" and section "数学公式" of the
 * euno.news page).  Device pointers: o_parts [C, T_q, H_q, 64] bf16 (the
 * chunks' out, stacked), o_residual_parts likewise or NULL, lse_parts
 * [C, H_q, T_q] fp32, sink [H_q] fp32; writes out [T_q, H_q, 64] bf16, its
 * optional residual out_residual, and lse [H_q, T_q] (-inf with out = 0 when
 * no chunk has a visible key and the sink is -inf).  head_dim must be 64
 * (ATTN_SINK_ERR_UNSUPPORTED otherwise); num_chunks >= 1, heads_q >= 1 and
 * 16-byte aligned tensors, else ATTN_SINK_ERR_INVALID_ARG.  total_q = 0 is a
 * no-op.  The merge runs in fp32.
 */
int attn_sink_merge(int num_chunks, int total_q, int heads_q, int head_dim, const void* o_parts,
                    const void* o_residual_parts, const float* lse_parts, const float* sink,
                    void* out, void* out_residual, float* lse, void* stream);

/*
 * Decode step over a paged key/value cache (one new query token per sequence):
 * the rollout-side forward with the same sink semantics as attn_sink_fwd, so
 * that inference and training compute the same log-probabilities (ai-engineering-
 * academy page, sections "Desafio 2: Inconsistência Treino-Inferência" and
 * "Desafio 3: Attention Sinks no FlashAttention"; the concat listing
 * "带汇聚的注意力（GPT-OSS）" of the euno.news page with one query row).
 */
typedef struct attn_sink_decode_params {
  int batch;          /* B >= 0 sequences */
  int heads_q;        /* H_q = G * heads_kv with G in {1, 2, 4, 8} (else UNSUPPORTED) */
  int heads_kv;       /* H_kv >= 1 */
  int head_dim;       /* must be 64 */
  int page_size;      /* keys per cache page, >= 1 */
  int num_pages;      /* pages in the cache pool */
  int max_pages;      /* columns of block_table (pages per sequence at most) */
  int window;         /* <= 0: every cached key; W > 0: the last W keys */
  float softmax_scale;/* multiplies q.k only; finite and > 0 */
} attn_sink_decode_params;

/*
 * Bytes of device workspace attn_sink_decode needs (0 if the params are
 * invalid or batch = 0): the key-split partial results and a completion
 * counter per (sequence, kv head), zeroed by the call before its one kernel
 * launch (the last split of each pair merges the partials with the sink).
 */
size_t attn_sink_decode_workspace_size(const attn_sink_decode_params* params);

/*
 * q [B, H_q, 64] bf16 (the new token of each sequence); k_cache, v_cache
 * [num_pages, page_size, H_kv, 64] bf16; block_table [B, max_pages] int32 (the
 * page of keys [p * page_size, (p + 1) * page_size) of sequence b);
 * seq_lens [B] int32, the cached keys of each sequence including the new
 * token's own (appended before the call); sink [H_q] fp32.  Writes out
 * [B, H_q, 64] bf16, optional out_residual (as attn_sink_fwd) and lse [H_q, B]
 * fp32; a sequence with no cached key gets out = 0, lse = sink.  The scores
 * multiply the bf16 inputs exactly with fp32 accumulation and the softmax runs
 * in fp32; P and v enter the P v product as fp16, as in attn_sink_fwd (v values
 * outside the fp16 range are reported as 0x400).  Block-table entries
 * and lengths are checked on the device (see attn_sink_device_error).  All
 * pointers are device pointers, 16-byte aligned where they hold bf16 rows;
 * the workspace is 256-byte aligned and at least
 * attn_sink_decode_workspace_size bytes.  batch and heads_kv above 65535
 * (launch-grid limits) return ATTN_SINK_ERR_UNSUPPORTED.  Returns an
 * attn_sink_status.
 */
int attn_sink_decode(const attn_sink_decode_params* params, const void* q, const void* k_cache,
                     const void* v_cache, const int* block_table, const int* seq_lens,
                     const float* sink, void* out, void* out_residual, float* lse,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * Flags of attn_sink_fwd_ex / attn_sink_bwd_ex, for a sink held as a bf16
 * training parameter whose gradient accumulates over micro-batches (direct use
 * under sharded data-parallel training; the pages train GPT-OSS with FSDP:
 * ai-engineering-academy page, section "Desafio 2: Inconsistência
 * Treino-Inferência").
 */
#define ATTN_SINK_FLAG_SINK_BF16 1        /* sink and dsink are bf16 [H_q] */
#define ATTN_SINK_FLAG_ACCUMULATE_DSINK 2 /* bwd: dsink += gradient (else =) */
#define ATTN_SINK_FLAG_DETERMINISTIC 4    /* bwd: as attn_sink_bwd_deterministic */

/*
 * attn_sink_fwd with flags (only ATTN_SINK_FLAG_SINK_BF16; any other bit
 * returns ATTN_SINK_ERR_INVALID_ARG).  With it, sink points to bf16 [H_q],
 * read exactly (bf16 -> fp32).  Everything else as attn_sink_fwd.
 */
int attn_sink_fwd_ex(const attn_sink_params* params, int flags, const void* q, const void* k,
                     const void* v, const void* sink, const int* cu_seqlens_q,
                     const int* cu_seqlens_k, void* out, void* out_residual, float* lse,
                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_sink_bwd with flags.  ATTN_SINK_FLAG_SINK_BF16: sink and dsink are bf16
 * [H_q] (dsink rounded to nearest from the fp32 sum);
 * ATTN_SINK_FLAG_ACCUMULATE_DSINK: dsink += the gradient (in fp32 for an fp32
 * dsink, in bf16 after the fp32 sum otherwise) instead of dsink = gradient;
 * ATTN_SINK_FLAG_DETERMINISTIC: the bitwise-reproducible backward.  Unknown
 * bits return ATTN_SINK_ERR_INVALID_ARG.  Everything else as attn_sink_bwd.
 */
int attn_sink_bwd_ex(const attn_sink_params* params, int flags, const void* q, const void* k,
                     const void* v, const void* sink, const int* cu_seqlens_q,
                     const int* cu_seqlens_k, const void* out, const void* out_residual,
                     const float* lse, const void* dout, void* dq, void* dk, void* dv,
                     void* dsink, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Bytes of device workspace attn_sink_fwd needs (0 if the params are invalid):
 * an fp16 copy of v [T_k, H_kv, 64] for the tensor cores and, for a packed
 * batch of two or more sequences, a table of its query tiles in the order the
 * forward runs them (heaviest first across sequences; 4 bytes a tile).  Same
 * conventions as attn_sink_bwd_workspace_size (packed fields when num_seqs >
 * 0).  A workspace that is missing, too small or not 256-byte aligned returns
 * ATTN_SINK_ERR_WORKSPACE.
 */
size_t attn_sink_fwd_workspace_size(const attn_sink_params* params);

/*
 * Size of the static scratch array behind attn_sink_fwd_noalloc: 16 MiB per
 * GPU that loads the library, held until the process exits.
 */
#define ATTN_SINK_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * Forward without a caller-provided workspace, for callers that cannot call
 * cudaMalloc themselves: code that runs inside a host framework which owns all
 * device memory through its own pool, or a latency-critical service that must
 * not allocate once it is running (cudaMalloc can synchronise the device and
 * fragment memory).  (The pages this library follows have no counterpart of
 * this entry point; it is a deployment convenience.)
 *
 * Same arguments, layouts and results as attn_sink_fwd, minus the workspace.
 * The scratch it needs (attn_sink_fwd_workspace_size bytes: the fp16 copy of v
 * and the tile order)
 * lives in a file-scope device array of ATTN_SINK_NOALLOC_SCRATCH_BYTES; a
 * problem that needs more returns ATTN_SINK_ERR_WORKSPACE and launches nothing.
 * The call allocates nothing.
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it; make that first call before any stream
 * capture.  The cached address belongs to the device's primary context:
 * resetting that context (cudaDeviceReset) after the first call is not
 * supported, since later calls would pass the old address.  Every call on a device shares the one array: calls that overlap on
 * the GPU (different streams, no ordering between them) race on it and must
 * be serialised by the caller.  Nothing in the array needs to start at zero:
 * each call overwrites the part it reads.
 */
int attn_sink_fwd_noalloc(const attn_sink_params* params, const void* q, const void* k,
                          const void* v, const float* sink, const int* cu_seqlens_q,
                          const int* cu_seqlens_k, void* out, void* out_residual, float* lse,
                          void* stream);

/*
 * Bytes of device workspace attn_sink_bwd needs for these params (0 if the
 * params are invalid).  The packed fields are used when num_seqs > 0, the
 * dense ones otherwise.  The workspace holds the row terms D [H_q, T_q], the
 * per-block dsink partials, the fp32 dq accumulator [T_q, H_q, 64] (bf16 dq
 * only), fp16 copies of q, dout, k and v, and, when the backward splits a GQA
 * group over several CTAs (decided from the shapes and the current device's SM
 * count), fp32 dK/dV partials, and for a packed batch of two or more
 * sequences a table of its key tiles in the order the backward runs them.
 * Query it on the device the backward will run on.
 */
size_t attn_sink_bwd_workspace_size(const attn_sink_params* params);

/*
 * Backward.  Reads q, k, v, sink, out (and optionally out_residual) and lse from
 * the forward and dout; writes dq, dk, dv (bf16 or fp32 per grad_dtype) and
 * dsink [H_q] fp32.  dk and dv sum over the query heads of each group.  dq, dk,
 * dv and dsink are overwritten.  dsink is reduced in a fixed order (bitwise
 * reproducible); dk and dv are too; dq is accumulated with fp32 atomics and may
 * differ in the last bits between runs.
 * Arithmetic: the five products run on fp16 copies of q, k, v, dout made in the
 * workspace (exact for |x| <= 65504; beyond it the device error word records
 * 0x400), with P and dS rounded to fp16 and fp32 accumulation.
 * Passage: section "反向传播" of the euno.news page for dsink.
 * Returns an attn_sink_status.
 */
int attn_sink_bwd(const attn_sink_params* params, const void* q, const void* k,
                  const void* v, const float* sink, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, const void* out, const void* out_residual,
                  const float* lse, const void* dout, void* dq, void* dk, void* dv,
                  float* dsink, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The backward of attn_sink_bwd with bitwise reproducible results: identical
 * inputs give identical dq, dk, dv and dsink on every call.  attn_sink_bwd
 * sums each query row's dQ over the key tiles with reduce-adds whose order the
 * hardware picks; here dQ comes from a separate query-stationary kernel that
 * recomputes S and dP and sums the key tiles in increasing order (two more
 * matrix products: about 40 % more arithmetic).  Train/inference consistency
 * and reproducibility are the pages' central lesson (keryc.com page on GPT-OSS
 * agentic RL fixes, section "Solutions implemented by the team"; euno.news
 * page, section "反向传播" for the gradient itself).  Arguments, layouts,
 * workspace (attn_sink_bwd_workspace_size covers both entry points), precision
 * and errors as attn_sink_bwd.
 */
int attn_sink_bwd_deterministic(const attn_sink_params* params, const void* q, const void* k,
                                const void* v, const float* sink, const int* cu_seqlens_q,
                                const int* cu_seqlens_k, const void* out,
                                const void* out_residual, const float* lse, const void* dout,
                                void* dq, void* dk, void* dv, float* dsink, void* workspace,
                                size_t workspace_bytes, void* stream);

/* Static, human-readable name of a status code. */
const char* attn_sink_status_string(int status);

/*
 * Synchronises `stream`, then reads and clears the device error word.  *code
 * receives 0 when nothing was recorded, 0x1xx / 0x2xx when a forward / backward
 * kernel gave up on a bounded wait, 0x400 when an input was outside the fp16
 * range of the tensor-core operands, 0x800 when attn_sink_decode met a
 * block-table entry outside [0, num_pages) or a sequence length outside
 * [0, max_pages * page_size] (that key is skipped; the length is clamped).
 * Only the first code recorded since the last read is kept.
 * The word is one per device, shared by every stream and every caller of the
 * library on that device: it is not tied to `stream`, so a code may come from
 * a launch on another stream, and a read clears it for every caller.  Callers
 * that run the library on several streams at once should read it after
 * synchronising all of them.
 * Returns ATTN_SINK_ERR_TIMEOUT when *code is a bounded-wait code (0x1xx or
 * 0x2xx), ATTN_SINK_ERR_CUDA when the synchronisation or the read itself
 * failed, ATTN_SINK_OK otherwise (including the input codes 0x400 / 0x800,
 * which *code reports).
 */
int attn_sink_device_error(void* stream, int* code);

/*
 * Number of kernels this library has launched in this process so far (a
 * host-side counter, incremented after every successful launch).  The
 * difference across a region counts the library's GPU launches in it.
 */
unsigned long long attn_sink_launch_count(void);

/*
 * The cudaError_t value of the most recent failed kernel launch of this
 * library in this process (0 when none failed), to explain an
 * ATTN_SINK_ERR_CUDA status.
 */
int attn_sink_last_cuda_error(void);

/*
 * Measurement hooks (no counterpart in the papers: they time this library's
 * own kernels).  Kernel ids for attn_sink_kernel_time:
 */
#define ATTN_SINK_KERNEL_FWD 0      /* the forward kernel: attn_sink_fwd_kernel or, for a
                                       sliding window, attn_sink_fwd_band_kernel */
#define ATTN_SINK_KERNEL_BWD_MAIN 1 /* attn_sink_bwd_main_kernel (all five backward products;
                                       without dQ under attn_sink_bwd_deterministic) */
#define ATTN_SINK_KERNEL_BWD_DQ 2   /* attn_sink_bwd_dq_kernel (attn_sink_bwd_deterministic) */
#define ATTN_SINK_KERNEL_MERGE 3    /* attn_sink_merge_kernel (attn_sink_merge) */
#define ATTN_SINK_KERNEL_COUNT 4

/*
 * on != 0: from now on every launch of the kernels above is bracketed by a
 * pair of CUDA events recorded on the launching stream (the events belong to
 * the library and are reused); on == 0 stops that.  Off at load.  Always
 * returns ATTN_SINK_OK.
 */
int attn_sink_kernel_timing(int on);

/*
 * Waits for every bracketed launch recorded so far, then writes the summed
 * duration in milliseconds (*total_ms) and the number of launches (*launches)
 * of `kernel` since the previous read of that kernel, and resets both.
 * ATTN_SINK_ERR_INVALID_ARG for a bad id or null pointer; ATTN_SINK_ERR_CUDA
 * if an event could not be read (those launches are left out of the sums).
 */
int attn_sink_kernel_time(int kernel, double* total_ms, unsigned long long* launches);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_SINK_H */
