// internal.h -- declarations shared by the C-ABI layer and the kernel translation units.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace ea46 {

// Per-launch parameters of the attention kernels (plain values and device pointers).
struct AttnParams {
  int B, H, S;
  int nQB;              // query blocks of 128 * NT rows per (b, h)
  int nK;               // key tiles of 128 = ceil(S / 128) = scale blocks per (b, h)
  float c_log2;         // softmax scale * log2(e)
  void* o;              // [B, S, H, D] bf16
  float* lse;           // [B, H, S] fp32 or nullptr
  const float* q_scale; // [B, H, nK] fp32 (FP8 only; nullptr = 1)
  const float* k_scale;
  const float* v_scale;
  long long spin_limit; // cycles a bounded wait may spin
  int* err_word;        // device error word (first error code)
  int* err_info;        // where it happened
  // packed variable-length batch (the VARLEN kernels): S = total tokens, B = 1
  const int* cu_seqlens; // [n_seq + 1] token offsets of the sequences
  int n_seq;
  int max_seqlen;        // bound on every sequence's length (checked by the kernel)
  int n_levels;          // ceil(max_seqlen / query rows per CTA)
  // grouped-query attention: query head h reads key/value head h / kv_group (1 = plain)
  int kv_group;
  // VARLEN with FP8: scale entries per head (total / 128 + n_seq + 1); the scale blocks of
  // sequence s start at index cu[s] / 128 + s
  int scale_stride;
};

// Key-split tail of a fixed-length, non-causal launch (n_parts <= 1: none).  Items
// 0 .. n_whole-1 are whole query blocks; item n_whole + part * n_tail + slot is key range
// `part` of query block n_whole + slot.  Scratch, device memory:
struct SplitParams {
  int n_whole, n_tail, n_parts;
  float* part_o;        // [n_tail][n_parts][128 NT rows][D] fp32 partial O (normalised)
  float* part_l;        // [n_tail][n_parts][128 NT rows] fp32 partial lse, log2 units
};

// At most this many key ranges per split tail block, each of at least KEY_SPLIT_MIN_TILES tiles.
constexpr int KEY_SPLIT_MAX_PARTS = 4;
constexpr int KEY_SPLIT_MIN_TILES = 4;
// Cost model of the plan, in key tiles: an item's fixed cost, and the merge's.
constexpr int KEY_SPLIT_ITEM_TILES = 4;
constexpr int KEY_SPLIT_MERGE_TILES = 4;


// Sequences and query-block levels a variable-length launch may hold: each CTA keeps the
// offsets, the sequences sorted by length and per-level counts in shared memory.
constexpr int VARLEN_MAX_SEQ = 4096;
constexpr int VARLEN_MAX_LEVELS = 1024;

// Launch one attention forward.  Returns the cudaError_t of the launch.
// `to` is O's bf16 map with a box of 32 columns x 32 rows and a 64-byte swizzle (the epilogue's
// tensor stores; unused by the packed-batch kernels).  `split` (fixed length, not causal; may be
// null) plans a key-split tail.
template <int D, bool FP8, bool CAUSAL, bool VARLEN = false>
cudaError_t launch_attn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& to, const AttnParams& p, cudaStream_t stream,
                        const SplitParams* split);

// Query-tile count per CTA (two Q tiles share K/V loads; one at D = 256 where
// two tiles' S and O would not fit the 512 Tensor-Memory columns).
constexpr int attn_q_tiles(int D) { return D == 256 ? 1 : 2; }

// Decoding with grouped key/value heads (attn_decode.cu).
struct DecodeParams {
  int B, Hq, Hkv, G, Sq, Sk;
  float c_log2;         // softmax scale * log2(e)
  void* o;              // [B, Sq, Hq, D] bf16
  float* lse;           // [B, Hq, Sq] fp32 or nullptr
  float* ws_o;          // [n_split][rows_total][D] fp32 partial outputs (n_split > 1)
  float* ws_l;          // [n_split][rows_total] fp32 partial lse
  int n_split;          // key splits per (b, key/value head)
  int tiles_per_split;  // 128-key tiles per split
  long long rows_total; // B * Hq * Sq
  long long spin_limit;
  int* err_word;
  int* err_info;
  // FP8 (E4M3 inputs): block scales as the quantiser writes them, or nullptr = 1
  const float* q_scale; // [B, Hq, nqb]
  const float* k_scale; // [B, Hkv, nkb]
  const float* v_scale; // [B, Hkv, nkb]
  int nqb, nkb;         // ceil(Sq / 128), ceil(Sk / 128)
};

// tq: the 5-D [B, Sq, Hkv, G, D] view of Q (box {one panel, G, 1, Sq, 1}); tk, tv: [B, Sk, Hkv, D].
cudaError_t launch_attn_decode(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeParams& p, int D, bool fp8, bool causal, cudaStream_t st);

// Backward pass (attn_bwd.cu).
struct BwdParams {
  int B, H, S;          // H: query heads
  int Hkv;              // key/value heads (H a multiple of Hkv; query head h reads h / (H / Hkv))
  int Sp;               // S rounded up to 128: row stride of the workspace
  float c_log2;         // softmax scale * log2(e)
  float scale;          // softmax scale
  const void* o;        // [B, S, H, D] bf16, the forward output
  const void* dout;     // [B, S, H, D] bf16
  const float* lse;     // [B, H, S] fp32, the forward's log-sum-exp
  float* ws;            // [B*H][2][Sp] fp32: Delta, lse*log2(e)
  void* dq;             // [B, S, H, D] bf16 outputs
  void* dk;             // [B, S, Hkv, D] bf16
  void* dv;
  long long spin_limit;
  int* err_word;
  int* err_info;
};

// Size of the fixed per-GPU scratch used by attn_bwd_noalloc, and its device address on the
// current GPU (looked up once per device; attn_bwd_noalloc.cu).
constexpr size_t NOALLOC_BWD_SCRATCH_BYTES = size_t(16) << 20;
cudaError_t noalloc_bwd_scratch(float** out);

// Delta kernel, dK/dV kernel, dQ kernel on `st`.  maps = Q, K, V, dO (bf16 maps: Q and dO over H
// heads, K and V over Hkv).
cudaError_t launch_attn_bwd(const CUtensorMap* maps, const BwdParams& p, int D, bool causal, cudaStream_t st);

struct QuantParams {
  int B, H, S, nblk;
  void* out;            // [B, S, H, D] E4M3
  float* scale;         // [B, H, nblk]
  const float* signs;   // [D] or nullptr
  const float* rope_cs; // [>= 128 * nblk, D/2, 2] rotary table (cos, sin of p * theta_i) or nullptr
  long long spin_limit; // cycles a bounded wait may spin
  int* err_word;        // device error word
  int* err_info;
  // packed variable-length batch (B = 1, S = total tokens): blocks of 128 tokens start at
  // every sequence's first token; block k of sequence s has scale index cu[s] / 128 + s + k,
  // nblk = total / 128 + n_seq + 1 indices per head (scale [H, nblk]); nullptr = fixed length
  const int* cu_seqlens;
  int n_seq;
  int n_pos;            // rows of rope_cs (VARLEN: checked against every sequence on the device)
  // Q, K and V in one launch (fixed length, no RoPE): tensor t's blocks follow tensor t-1's,
  // its scales go to scale (t = 0), scale1, scale2, and the first rot_tensors are rotated
  int n_tensors = 1;
  int rot_tensors = 1;
  float* scale1 = nullptr;
  float* scale2 = nullptr;
};

// Tensor maps of the quantiser's inputs and outputs: [0] only, or Q, K, V.
struct QuantMaps {
  CUtensorMap x[3];
  CUtensorMap out[3];
};

// x is read through `tx`, the same [B, S, H, D] bf16 tensor map the attention kernel uses;
// codes are written through `tout`, an E4M3 map of the same tensor whose box is one warp's
// rows (32, or 16 at D = 256).
template <int D>
cudaError_t launch_hadamard_quant(const QuantMaps& m, const QuantParams& p,
                                  cudaStream_t stream);

// cs[p, i] = (cos, sin)(p * base^(-2i/D)) for p < n_pos, i < D/2, in fp64 rounded to fp32.
cudaError_t launch_rope_table(float* cs, int n_pos, int D, double base, cudaStream_t stream);

}  // namespace ea46
