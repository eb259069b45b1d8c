/*
 * attn46.h -- C ABI of the fused exact-attention forward library for GB300 (sm_103a).
 *
 * The library computes, on one GPU, the attention forward pass
 *
 *     O = softmax(scale * Q K^T [+ causal mask]) V,   lse = log-sum-exp per query row,
 *
 * tile by tile with an online softmax, never writing the S x S score matrix to
 * device memory, and the low-precision variant in which Q and K are first
 * rotated by a random-sign Hadamard matrix and Q, K, V are quantised to FP8
 * (E4M3) with one scale per 128-token block.
 *
 * Sources (web pages, cited by title and section):
 *   [HADA] "FlashAttention-3: Schnellere und präzisere Attention durch
 *          Asynchronität und geringe Präzision" (hada.io summary of the FA3
 *          announcement);
 *   [NL]   "FlashAttention-3 (NL)" (systems-analysis.info).
 *
 * Conventions shared by every entry point:
 *   - Pointers named q, k, v, o, x, out, lse, *_scale, signs are DEVICE
 *     pointers owned by the caller; the library never frees or keeps them.
 *   - Tensor layout is [B, S, H, D] contiguous (one row = one token of one
 *     head, D contiguous elements); lse is [B, H, S] fp32; block scales are
 *     [B, H, ceil(S/128)] fp32.  q, k, v, o, x and out must be 16-byte aligned.
 *   - stream is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls only enqueue work and return; they do not synchronise.
 *   - Return value: an attn_status.  On any non-OK status nothing was launched
 *     and attn_get_last_error() describes why.  Device-side failures (a
 *     bounded wait inside a kernel that ran out) are recorded in a per-device
 *     error word and reported by attn_check().
 *   - No C++ exception crosses this boundary.
 *   - B, H, S >= 1; D in {64, 128, 256}; outputs must not overlap inputs.
 */
#ifndef ATTN46_H
#define ATTN46_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, bad size, overlap, bad enum */
  ATTN_ERR_UNSUPPORTED = 2,   /* valid request this build does not implement (e.g. D = 96) */
  ATTN_ERR_CUDA = 3,          /* a CUDA runtime or driver call failed */
  ATTN_ERR_TIMEOUT = 4        /* a bounded wait inside a kernel ran out (see attn_check) */
} attn_status;

typedef enum {
  ATTN_BF16 = 0,              /* q, k, v bf16 */
  ATTN_FP8_E4M3 = 1           /* q, k, v E4M3 bytes with unit scales */
} attn_dtype;

/*
 * attn_fwd -- fused exact attention forward.
 *   [HADA] "Rückblick auf den FlashAttention-Ansatz": blocks of the inputs are
 *   loaded on chip, attention is computed per block with softmax rescaling,
 *   and the exact output is obtained without writing the attention matrix to
 *   HBM; "Überlappung von GEMM und Softmax": the work is the Q-K GEMM, the
 *   softmax and the P-V GEMM.
 *   q, k, v : [B, S, H, D] bf16 (dtype ATTN_BF16) or E4M3 (ATTN_FP8_E4M3, all
 *             scales taken as 1).
 *   o       : [B, S, H, D] bf16 output.
 *   lse     : [B, H, S] fp32 natural-log log-sum-exp of the scaled, masked
 *             logits, or NULL to skip it.
 *   causal  : 0 = every query sees every key; 1 = query i sees keys j <= i.
 *   scale   : logit multiplier; 0 selects 1/sqrt(D); negative or non-finite
 *             values are rejected.
 *   Scheduling: one persistent CTA per SM walks the query blocks.  attn_fwd,
 *   attn_fwd_fp8, attn_fwd_gqa and attn_fwd_gqa_fp8 allocate nothing and
 *   always run every block whole; the key-split tail (cutting the blocks of
 *   a partly filled last round into key ranges) needs scratch and is
 *   attn_fwd_split's, with a caller workspace.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int H, int S, int D, int causal, float scale, int dtype,
             void* stream);

/*
 * attn_fwd_fp8 -- attention forward on E4M3 inputs with per-block scales.
 *   [NL] "Technische innovaties", item 3, and [HADA] "Niedrige
 *   FP8-Präzision und incoherent processing": both GEMMs run in FP8; the
 *   inputs come from hadamard_rotate_quant_fp8.
 *   q8, k8, v8 : [B, S, H, D] E4M3 bytes; the value of an element is
 *                code * its block's scale.
 *   q_scale, k_scale, v_scale : [B, H, ceil(S/128)] fp32 scales, as written by
 *                hadamard_rotate_quant_fp8 (which never writes 0).  Scales must be
 *                finite; Q and K scales positive, V scales >= 0 (a 0 block holds
 *                zeros: it adds nothing to O and its keys still count in lse).
 *   o, lse, causal, scale : as for attn_fwd (scale refers to the original
 *                head dimension; the rotation does not change it).
 *   The softmax numerators are rounded to E4M3 for the P-V GEMM; the row sums
 *   use the unrounded values.
 */
int attn_fwd_fp8(const void* q8, const void* k8, const void* v8,
                 const float* q_scale, const float* k_scale, const float* v_scale,
                 void* o, float* lse, int B, int H, int S, int D, int causal,
                 float scale, void* stream);

/*
 * attn_fwd_varlen -- attn_fwd over a packed batch of variable-length sequences.
 *   [HADA] "Weitere Optimierungen und künftige Integration" lists variable-
 *   length sequences among the paper's optimisations; the pages define
 *   nothing further.  Reading: the sequences are concatenated along one token
 *   axis and each attends only to itself (causal: to its own keys j <= i,
 *   positions counted from its first token).
 *   q, k, v, o : [total, H, D] bf16, contiguous, 16-byte aligned.
 *   lse        : [H, total] fp32, natural log, or NULL.
 *   cu_seqlens : device int32 [n_seq + 1]: cu_seqlens[0] = 0, non-decreasing,
 *                cu_seqlens[n_seq] = total; sequence s is tokens
 *                cu_seqlens[s] .. cu_seqlens[s+1]-1 (empty sequences allowed).
 *   n_seq      : 1 .. 4096.  total >= 1.  D in {64, 128, 256}.
 *   max_seqlen : a bound on every sequence's length, 1 .. 262144 (131072 at
 *                D = 256; larger is ATTN_ERR_UNSUPPORTED); it sizes the
 *                kernel's per-level work lists.
 *   Work is ordered heaviest first (the query blocks with the most keys, and
 *   the longest sequences), as in attn_fwd.
 *   Host-side checks as attn_fwd (ATTN_ERR_INVALID_ARG / _UNSUPPORTED, no
 *   launch).  cu_seqlens lives on the device, so its contents are checked by
 *   the kernel: offsets that break the rules above, or a sequence longer than
 *   max_seqlen, make the launch write nothing and leave ATTN_ERR_INVALID_ARG
 *   in the device error word, which attn_check() reports.
 */
int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                    const int* cu_seqlens, int n_seq, int total, int max_seqlen, int H, int D,
                    int causal, float scale, void* stream);

/*
 * The FP8 path on packed variable-length batches: the rotation and block
 *   quantisation of [HADA] "Niedrige FP8-Präzision und incoherent processing"
 *   with the packed batches of [HADA] "Weitere Optimierungen und künftige
 *   Integration".  Reading (the pages define neither the combination nor a
 *   layout): a scale block never straddles two sequences -- sequence s is cut
 *   into 128-token blocks from its own first token -- and the scales of all
 *   sequences share one array [H, NB], NB = attn_varlen_scale_blocks(total,
 *   n_seq) = total / 128 + n_seq + 1, block k of sequence s at index
 *   cu_seqlens[s] / 128 + s + k (indices no block uses are left unwritten).
 *
 * attn_varlen_scale_blocks -- NB above (0 for negative arguments).
 *
 * hadamard_rotate_quant_fp8_varlen -- hadamard_rotate_quant_fp8 on a packed
 *   batch: x [total, H, D] bf16 -> out [total, H, D] E4M3, scale [H, NB] fp32.
 *   cu_seqlens as attn_fwd_varlen (device int32 [n_seq + 1], n_seq 1..4096);
 *   offsets that are not 0 .. total, non-decreasing, make the launch write
 *   nothing and leave ATTN_ERR_INVALID_ARG for attn_check().  No RoPE fusion.
 *
 * attn_fwd_varlen_fp8 -- attn_fwd_varlen on E4M3 codes with those scales
 *   (q_scale, k_scale, v_scale [H, NB] fp32, non-null, 4-byte aligned); the
 *   value scales enter as in attn_fwd_fp8, with the largest taken over the
 *   sequence's own blocks.  Other arguments and errors as attn_fwd_varlen.
 */
int attn_varlen_scale_blocks(int total, int n_seq);
int hadamard_rotate_quant_fp8_varlen(const void* x, void* out, float* scale, const float* signs,
                                     const int* cu_seqlens, int n_seq, int total, int H, int D,
                                     void* stream);
/*
 * rope_hadamard_rotate_quant_fp8_varlen -- the same with rotary embedding in front
 *   (rope_hadamard_rotate_quant_fp8 on a packed batch): positions restart at
 *   every sequence's first token.  rope_cs as rope_cos_sin_table writes it,
 *   n_pos >= 128 rows; a sequence with 128 * ceil(len / 128) > n_pos is an error
 *   found on the device with the offsets check (nothing is written).
 */
int rope_hadamard_rotate_quant_fp8_varlen(const void* x, const float* rope_cs, int n_pos, void* out,
                                          float* scale, const float* signs, const int* cu_seqlens,
                                          int n_seq, int total, int H, int D, void* stream);
int attn_fwd_varlen_fp8(const void* q8, const void* k8, const void* v8, const float* q_scale,
                        const float* k_scale, const float* v_scale, void* o, float* lse,
                        const int* cu_seqlens, int n_seq, int total, int max_seqlen, int H, int D,
                        int causal, float scale, void* stream);

/*
 * attn_fwd_gqa -- attn_fwd (BF16) with grouped key/value heads.
 *   The pages name LLM inference as future work ([HADA] "Weitere
 *   Optimierungen und künftige Integration"); grouped-query attention is
 *   the reading: Hq query heads share Hkv key/value heads, query head h reads
 *   key/value head h / (Hq / Hkv).
 *   q, o : [B, S, Hq, D] bf16.   k, v : [B, S, Hkv, D] bf16.   lse [B, Hq, S].
 *   Hq a positive multiple of Hkv; other arguments and errors as attn_fwd.
 */
int attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                 int Hq, int Hkv, int S, int D, int causal, float scale, void* stream);

/*
 * attn_fwd_gqa_fp8 -- attn_fwd_fp8 with grouped key/value heads: the FP8 path of
 *   [HADA] "Niedrige FP8-Präzision und incoherent processing" with the grouping
 *   of attn_fwd_gqa.
 *   q8 : [B, S, Hq, D] E4M3 bytes, q_scale [B, Hq, ceil(S/128)] fp32.
 *   k8, v8 : [B, S, Hkv, D] E4M3 bytes, k_scale, v_scale [B, Hkv, ceil(S/128)]
 *   fp32 (the layout hadamard_rotate_quant_fp8 writes for each tensor).
 *   o : [B, S, Hq, D] bf16.   lse : [B, Hq, S] fp32 or NULL.
 *   Hq a positive multiple of Hkv; scales non-null and 4-byte aligned; other
 *   arguments and errors as attn_fwd_fp8.
 */
int attn_fwd_gqa_fp8(const void* q8, const void* k8, const void* v8, const float* q_scale,
                     const float* k_scale, const float* v_scale, void* o, float* lse, int B, int Hq,
                     int Hkv, int S, int D, int causal, float scale, void* stream);

/*
 * attn_decode -- attention of Sq query tokens against Sk >= Sq keys with
 *   grouped key/value heads: decoding (Sq = 1) and short query blocks.
 *   The queries are the last Sq positions: under the causal mask query i sees
 *   keys j <= Sk - Sq + i.  Query head h reads key/value head h / G, G = Hq / Hkv.
 *   q, o : [B, Sq, Hq, D] bf16.   k, v : [B, Sk, Hkv, D] bf16.
 *   lse  : [B, Hq, Sq] fp32 or NULL.
 *   D in {64, 128}; G * Sq <= 128 (the G heads x Sq tokens of one key/value
 *   head share one 128-row tile; ATTN_ERR_UNSUPPORTED otherwise).
 *   The keys are split over CTAs to fill the GPU; with more than one split
 *   the partial results go to `workspace` (caller-owned device scratch of
 *   attn_decode_workspace_bytes(...) bytes, 16-byte aligned, overwritten; it
 *   may be NULL when that function returns 0) and a second kernel merges
 *   them.  The split count depends on the shape and the current device's SM
 *   count only.
 */
size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D);
int attn_decode(const void* q, const void* k, const void* v, void* o, float* lse, float* workspace,
                size_t workspace_bytes, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal,
                float scale, void* stream);

/*
 * attn_decode_fp8 -- attn_decode on E4M3 inputs with per-block scales: the
 *   FP8 path of [HADA] "Niedrige FP8-Präzision und incoherent processing"
 *   (block quantisation of the rotated Q and K) applied to a decoding step,
 *   so that a step streams one byte per cached element instead of two.
 *   q8   : [B, Sq, Hq, D] E4M3 bytes.   k8, v8 : [B, Sk, Hkv, D] E4M3 bytes.
 *   q_scale : [B, Hq, ceil(Sq/128)] fp32; k_scale, v_scale : [B, Hkv,
 *             ceil(Sk/128)] fp32; an element's value is code * its block's
 *             scale -- the layout hadamard_rotate_quant_fp8 writes, so the
 *             key/value cache is quantised by (b, key/value head, 128-token
 *             block).  All three non-null, 4-byte aligned, device memory.
 *   Q and K rotated by the same signs (or neither) give the same logits.
 *   o, lse, workspace (attn_decode_workspace_bytes), shapes, the mask and the
 *   errors as attn_decode.  The numerators of P reach the tensor core as E4M3,
 *   as in attn_fwd_fp8.
 */
int attn_decode_fp8(const void* q8, const void* k8, const void* v8, const float* q_scale,
                    const float* k_scale, const float* v_scale, void* o, float* lse, float* workspace,
                    size_t workspace_bytes, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal,
                    float scale, void* stream);

/*
 * attn_bwd -- gradients dQ, dK, dV of attn_fwd (BF16), recomputed from the saved
 * log-sum-exp.
 *   The pages describe FlashAttention as tiling plus recomputation ([HADA]
 *   "Rückblick auf den FlashAttention-Ansatz"): the score matrix is never
 *   stored; the backward recomputes it tile by tile.  With
 *   P = exp(scale * Q K^T - lse) (masked): dV = P^T dO, dP = dO V^T,
 *   Delta_i = sum_d dO_id O_id, dS = P * (dP - Delta), dQ = scale * dS K,
 *   dK = scale * dS^T Q.
 *   q, k, v, o, dout : [B, S, H, D] bf16 inputs (o = attn_fwd's output).
 *   lse              : [B, H, S] fp32, attn_fwd's log-sum-exp for the same
 *                      q, k, v, causal flag and scale.
 *   dq, dk, dv       : [B, S, H, D] bf16 outputs.
 *   workspace        : device scratch of workspace_bytes >= attn_bwd_workspace_bytes(B, H, S)
 *                      (per row: Delta and lse * log2(e)); owned by the
 *                      caller, contents overwritten.
 *   D in {64, 128} (256: ATTN_ERR_UNSUPPORTED).  causal, scale as attn_fwd.
 *   Three kernels on `stream`: Delta, then dK/dV, then dQ.  Alignment 16 bytes
 *   (lse 4); outputs and workspace must not overlap inputs or each other.
 */
size_t attn_bwd_workspace_bytes(int B, int H, int S);
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, float* workspace,
             size_t workspace_bytes, int B, int H, int S, int D, int causal, float scale,
             void* stream);

/*
 * attn_bwd_gqa -- attn_bwd for grouped-query attention: the gradients of
 *   attn_fwd_gqa (Hq query heads over Hkv key/value heads, query head h
 *   reading key/value head h / (Hq / Hkv)).  This is the backward of
 *   multi-head attention with each key/value head repeated over its group of
 *   G = Hq / Hkv query heads; dQ is that backward's dQ, and dK, dV of a
 *   key/value head are the sums of the repeated heads' dK, dV over the group.
 *   q, o, dout : [B, S, Hq, D] bf16.   k, v : [B, S, Hkv, D] bf16.
 *   lse        : [B, Hq, S] fp32 (attn_fwd_gqa's).
 *   dq         : [B, S, Hq, D] bf16 output; dk, dv : [B, S, Hkv, D] bf16.
 *   workspace  : workspace_bytes >= attn_bwd_workspace_bytes(B, Hq, S).
 *   Hq a positive multiple of Hkv, else ATTN_ERR_INVALID_ARG; Hkv = Hq gives
 *   exactly attn_bwd.  Everything else as attn_bwd.  The group's sum is
 *   formed in fp32 inside one CTA per (128 keys, b, key/value head) and
 *   rounded to bf16 once.
 */
int attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, float* workspace,
                 size_t workspace_bytes, int B, int Hq, int Hkv, int S, int D, int causal,
                 float scale, void* stream);

/*
 * attn_bwd_noalloc -- attn_bwd without a caller workspace.  The paper has no
 *   counterpart; this is a convenience of this library.
 *   For callers that cannot allocate device memory where they run the
 *   backward pass: an engine that gave nearly all of the GPU's memory to its
 *   own pool at start-up, or a host that forbids allocation inside per-step
 *   calls, cannot get a fresh workspace buffer.  This entry point uses a
 *   fixed 16 MiB scratch array that the library carries on every GPU that
 *   loads it (held until the process exits); no call allocates or frees.
 *   Arguments, layouts, results and errors as attn_bwd, minus the workspace.
 *   Limit: attn_bwd_workspace_bytes(B, H, S) <= 16 MiB, i.e.
 *   B * H * (S rounded up to 128) <= 2,097,152; larger problems are rejected
 *   with ATTN_ERR_INVALID_ARG before anything runs.
 *   Every call looks up the scratch's device address (cudaGetSymbolAddress)
 *   with the caller's device current -- a host-side query, nothing is
 *   allocated; make the first call on a device before any stream capture, as
 *   that first lookup loads the library's device code there.  All calls on a
 *   device share the scratch and
 *   it keeps the last call's contents (every call rewrites what it reads, so
 *   nothing needs clearing); calls whose kernels overlap on the GPU race on
 *   it and may give wrong gradients, so serialise them.
 */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, int B, int H, int S, int D,
                     int causal, float scale, void* stream);

/*
 * hadamard_rotate_quant_fp8 -- random-sign Hadamard rotation + blockwise E4M3 quantisation.
 *   [NL] "Technische innovaties", item 3, steps 1-3: multiply by a random
 *   orthogonal matrix, which spreads outliers over the coordinates, then
 *   quantise to FP8.  [HADA] "Niedrige FP8-Präzision und incoherent
 *   processing": a Hadamard transform with random signs, O(d log d) per
 *   head, memory-bandwidth bound.
 *   x      : [B, S, H, D] bf16 input.
 *   out    : [B, S, H, D] E4M3 bytes.
 *   scale  : [B, H, ceil(S/128)] fp32 output; scale = amax / 448 of the
 *            block's rotated values (1 for an all-zero block).
 *   signs  : D fp32 values, each +1 or -1, or NULL to quantise without
 *            rotating.  Each row x (D elements) becomes
 *            x' = (x * signs) H_D / sqrt(D), H_D the Sylvester Hadamard
 *            matrix; use the same signs for Q and K.
 *   out[e] = E4M3_round_nearest_even_saturating(x'[e] / scale).
 *   Ordering: the launch may start while the kernel before it on the stream
 *   is finishing (programmatic dependent launch), but only its set-up runs
 *   then: it reads no input before that kernel has completed and its writes
 *   are visible, so stream order holds for every argument.
 */
int hadamard_rotate_quant_fp8(const void* x, void* out, float* scale, const float* signs,
                              int B, int H, int S, int D, void* stream);

/*
 * hadamard_rotate_quant_fp8_qkv -- hadamard_rotate_quant_fp8 of Q and K
 * (rotated by the same signs) and of V (not rotated), in one launch.
 *   [NL] "Technische innovaties", item 3, and [HADA] "Niedrige FP8-Präzision
 *   und incoherent processing", as for hadamard_rotate_quant_fp8: the
 *   rotation is applied to the two operands of Q K^T, whose product it
 *   leaves unchanged; V is quantised as it is.
 *   q, k, v        : [B, S, H, D] bf16 inputs (16-byte aligned).
 *   q8, k8, v8     : [B, S, H, D] E4M3 outputs (16-byte aligned).
 *   q_scale, k_scale, v_scale : [B, H, ceil(S/128)] fp32 outputs.
 *   signs          : D fp32 values +1 / -1 for Q and K, or NULL (then none
 *                    of the three is rotated).
 *   Every output holds exactly what hadamard_rotate_quant_fp8 writes for
 *   its tensor (the same arithmetic); the three tensors' blocks are one
 *   grid's work list, so the launch has one start-up and one tail instead of
 *   three.  The six outputs must overlap neither each other nor the inputs.
 *   Ordering and errors as hadamard_rotate_quant_fp8.
 */
int hadamard_rotate_quant_fp8_qkv(const void* q, const void* k, const void* v, void* q8, void* k8,
                                  void* v8, float* q_scale, float* k_scale, float* v_scale,
                                  const float* signs, int B, int H, int S, int D, void* stream);

/*
 * rope_cos_sin_table -- the rotary-embedding table.
 *   [HADA] "Niedrige FP8-Präzision und incoherent processing" names rotary
 *   embedding as the bandwidth-bound op to fuse the rotation with but does
 *   not define it; the reading is RoFormer's (Su et al. 2021, section 3.2):
 *   pair (x[2i], x[2i+1]) of the row at position p turns by p * theta_i,
 *   theta_i = base^(-2i/D).
 *   cs     : device output, [n_pos, D/2, 2] fp32, cs[p][i] = (cos, sin) of
 *            p * theta_i, evaluated in fp64 and rounded to nearest fp32;
 *            8-byte aligned.
 *   n_pos  : positions 0 .. n_pos-1, 1 <= n_pos <= 2^26.
 *   D      : even, 2 .. 4096.  base: finite, > 0 (10000 in RoFormer).
 *   Enqueued on `stream`; the caller owns cs and normally builds it once.
 */
int rope_cos_sin_table(float* cs, int n_pos, int D, double base, void* stream);

/*
 * rope_hadamard_rotate_quant_fp8 -- rotary embedding fused into the
 * rotation + quantiser (the fusion [HADA] says makes the rotation free).
 *   Each row x of token s (position p = s) becomes
 *   x' = (rope_p(x) * signs) H_D / sqrt(D), in fp32 with no rounding in
 *   between, then is quantised exactly as by hadamard_rotate_quant_fp8
 *   (signs may be NULL: RoPE + quantiser only).  Apply to Q and K, not V.
 *   rope_cs: the table written by rope_cos_sin_table for this D and base,
 *            16-byte aligned, with n_pos >= 128 * ceil(S/128) rows.  The
 *            kernel reads rows 0..15 and the rows at multiples of 16 and
 *            rebuilds the others with the angle-addition identity, so the
 *            table must be a rotary table of that form.
 *   Other arguments, layouts and errors as hadamard_rotate_quant_fp8;
 *   ATTN_ERR_INVALID_ARG also for a null or short table.
 */
int rope_hadamard_rotate_quant_fp8(const void* x, const float* rope_cs, int n_pos, void* out,
                                   float* scale, const float* signs, int B, int H, int S, int D,
                                   void* stream);

/* Message for the last non-OK status returned on the calling host thread ("" if none). */
const char* attn_get_last_error(void);

/*
 * attn_check -- synchronise `stream`, then read and clear the current
 * device's error word.  Returns ATTN_OK, ATTN_ERR_TIMEOUT (a kernel's bounded
 * wait ran out; its outputs are undefined), ATTN_ERR_INVALID_ARG (a
 * variable-length launch found bad cu_seqlens; it wrote nothing) or
 * ATTN_ERR_CUDA.
 */
int attn_check(void* stream);

/*
 * attn_set_spin_limit -- cycles (SM clock) a kernel's bounded wait may spin
 * before it gives up and records ATTN_ERR_TIMEOUT; 0 restores the default
 * (about 4e9 cycles, two seconds at 2 GHz).  Applies to later launches from
 * any host thread.
 */
void attn_set_spin_limit(long long cycles);

/*
 * attn_fwd_split -- attn_fwd / attn_fwd_fp8 / attn_fwd_gqa / attn_fwd_gqa_fp8
 *   with a caller workspace for the key-split tail.  The pages have no
 *   counterpart ([HADA] "Weitere Optimierungen und künftige Integration"
 *   names the persistent kernel; how its last round is filled is this
 *   library's scheduling).
 *   Without the causal mask, when the B * Hq * ceil(S / (128 * tiles per CTA))
 *   query blocks do not fill the last round of persistent CTAs (one per SM),
 *   the blocks of that round may be cut into key ranges (attn_key_split_plan,
 *   at most attn_set_key_split's ranges); each range writes its normalised
 *   partial output (fp32) and lse to the workspace, and a second kernel on
 *   the same stream merges every cut row over its ranges in a fixed order.
 *   q, k, v, o, lse, B, S, D, causal, scale : as attn_fwd_gqa (Hq query heads,
 *             Hkv key/value heads, Hq a multiple of Hkv; Hkv = Hq is attn_fwd).
 *   q_scale, k_scale, v_scale : NULL for bf16 (dtype ATTN_BF16) and for E4M3
 *             codes with unit scales; all three non-null for E4M3 codes with
 *             block scales (layouts as attn_fwd_gqa_fp8).  One or two non-null
 *             is ATTN_ERR_INVALID_ARG.
 *   dtype   : ATTN_BF16 or ATTN_FP8_E4M3.
 *   workspace : caller-owned device scratch, 16-byte aligned, overwritten,
 *             overlapping no input or output; or NULL, which runs every block
 *             whole (the result of attn_fwd).  With a workspace, a problem the
 *             plan splits needs workspace_bytes >=
 *             attn_fwd_split_workspace_bytes(B, Hq, S, D, causal); less is
 *             ATTN_ERR_INVALID_ARG, never a silent fallback, so the same
 *             arguments always run the same launches and give the same bits.
 *   Rows of blocks that run whole are bitwise those of attn_fwd; rows of cut
 *   blocks differ by rounding only (each range rounds its softmax numerators
 *   against its own running maximum).
 */
int attn_fwd_split(const void* q, const void* k, const void* v, const float* q_scale,
                   const float* k_scale, const float* v_scale, void* o, float* lse, int B,
                   int Hq, int Hkv, int S, int D, int causal, float scale, int dtype,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_fwd_split_workspace_bytes -- the workspace attn_fwd_split needs for
 *   this shape on the current device (its SM count sets the plan) under the
 *   current attn_set_key_split limit: 4 * (D + 1) bytes per row of every cut
 *   range, 128 * (2, or 1 at D = 256) rows per range.  0 when the plan does
 *   not split (causal, a full last round, too few key tiles, or the split
 *   turned off) or for invalid arguments.
 */
size_t attn_fwd_split_workspace_bytes(int B, int Hq, int S, int D, int causal);

/*
 * attn_set_key_split -- the most key ranges a query block of the last,
 *   partly filled round of a non-causal forward may be cut into (see
 *   attn_fwd_split); clamped to [1, 4], 1 turns the split off, 4 is the default.
 *   Applies to later launches from any host thread.  The pages have no
 *   counterpart: this is a scheduling choice of this library.
 */
void attn_set_key_split(int max_parts);

/*
 * attn_key_split_plan -- the split a non-causal forward of n_items equal
 *   query blocks (B * H * ceil(S / (128 * tiles per CTA)); tiles per CTA = 2,
 *   or 1 at D = 256) with key_tiles = ceil(S / 128) gets on `sms` persistent
 *   CTAs with at most max_parts ranges per block.  Host only; no device call.
 *   out[0] = blocks run whole (a multiple of sms), out[1] = blocks cut,
 *   out[2] = ranges per cut block (1: no split).  Cost model, in key tiles
 *   (a block costs about 4 tiles beyond its own, and so does the merge):
 *   the last round costs key_tiles + 4 unsplit and, cut into s ranges,
 *   ceil(n_tail * s / sms) * (ceil(key_tiles / s) + 4) + 4, with
 *   n_tail = n_items mod sms.  The plan takes the cheapest s <= max_parts
 *   whose ranges have at least 4 key tiles, if it costs at most 85 % of the
 *   unsplit round; problems with no full round are not split.
 *   ATTN_ERR_INVALID_ARG if out is NULL, n_items < 0, sms < 1 or
 *   key_tiles < 0.
 */
int attn_key_split_plan(long long n_items, int sms, int key_tiles, int max_parts, long long* out);

/*
 * attn_selftest_bounded_wait -- launch one tiny kernel whose bounded wait
 * targets a barrier nothing ever completes, with the given spin limit, so
 * the timeout path can be checked without hanging or faulting the GPU.  The
 * kernel records ATTN_ERR_TIMEOUT and returns; attn_check() then reports it.
 */
int attn_selftest_bounded_wait(long long spin_cycles, void* stream);

/* Library ABI version (major * 100 + minor). */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN46_H */
