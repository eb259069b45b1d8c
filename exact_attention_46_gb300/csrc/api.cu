// api.cu -- the C ABI (include/attn46.h): argument checks, TMA descriptors, launches, the
// device error word and its readback.  No computation of the method happens here.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "attn46.h"
#include "internal.h"
#include "ptx.cuh"

namespace {

using namespace ea46;

thread_local char g_msg[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_msg[0] = '\0';
  return ATTN_OK;
}

std::atomic<long long> g_spin_limit{0};
constexpr long long kDefaultSpin = 4000000000LL;

long long spin_limit() {
  const long long v = g_spin_limit.load();
  return v > 0 ? v : kDefaultSpin;
}

// Device error word: [0] = first error code of the launches since the last attn_check,
// [1] = where it happened.  One copy per device (module-scope device variable).  Its address
// is looked up on every call, with the caller's device current: the lookup is a host query,
// not stream work, and an address kept from an earlier context (before a device reset) would
// be stale.
__device__ int g_err_word[2];

int err_words(int** out) {
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_err_word);
  if (e != cudaSuccess)
    return fail(ATTN_ERR_CUDA, "cudaGetSymbolAddress(error word): %s", cudaGetErrorString(e));
  *out = static_cast<int*>(ptr);
  return ATTN_OK;
}

// ---- TMA descriptor encoding through the driver entry point (no link-time libcuda) ----

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// [B, S, H, D] tensor viewed as the 4-D box grid (D, H, S, B); one box = 128 tokens x one
// swizzle panel of one head.
// L2 promotion no wider than one row: a row of another head sits beside each row, and a wider
// promotion would fetch it from HBM with this one.
CUtensorMapL2promotion l2_promotion(int row_bytes) {
  return row_bytes >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                          : (row_bytes >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_64B);
}

int make_qkv_map(CUtensorMap* m, const void* ptr, int B, int S, int H, int D, bool fp8, int box_rows = 128);

// O [B, S, H, D] bf16 for the forward's epilogue: a box of 32 columns x 32 rows (one softmax
// warp's rows, one 32-column chunk), 64-byte swizzle.
int make_o_map(CUtensorMap* m, const void* ptr, int B, int S, int H, int D) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2,
                                 static_cast<cuuint64_t>(S) * H * D * 2};
  const cuuint32_t box[4] = {32, 1, 32, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed for O (%d)", int(r));
  return ATTN_OK;
}

int make_qkv_map(CUtensorMap* m, const void* ptr, int B, int S, int H, int D, bool fp8, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  const int esz = fp8 ? 1 : 2;
  const int row_bytes = D * esz;
  const int panel_row = row_bytes >= 128 ? 128 : row_bytes;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * esz,
                                 static_cast<cuuint64_t>(H) * D * esz,
                                 static_cast<cuuint64_t>(S) * H * D * esz};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(panel_row / esz), 1, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         4, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE,
                         panel_row == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                         l2_promotion(row_bytes), CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// ---- key-split tail of the fixed-length, non-causal forward (attn_kernel.cuh) ----

std::atomic<int> g_key_split_max{KEY_SPLIT_MAX_PARTS};

struct SplitPlan {
  long long n_whole, n_tail;
  int n_parts;
};

// n_items equal items on `sms` persistent CTAs take ceil(n_items / sms) rounds, the last one
// partly idle.  Cutting each of its n_tail = n_items mod sms blocks into s key ranges makes it
// ceil(n_tail * s / sms) rounds of ranges of at most ceil(nK / s) key tiles.  Measured on
// GB300, an item costs about KEY_SPLIT_ITEM_TILES key tiles on top of its own (start and
// epilogue), and the merge about KEY_SPLIT_MERGE_TILES.  In key tiles, the last round costs
// nK + ITEM unsplit and ceil(n_tail s / sms) (ceil(nK / s) + ITEM) + MERGE split; the plan
// takes the cheapest s <= max_parts (every range at least KEY_SPLIT_MIN_TILES tiles) if it
// costs at most 85 % of the unsplit round.  Problems without one full round are not split.
SplitPlan key_split_plan(long long n_items, int sms, int nK, int max_parts) {
  SplitPlan sp{n_items, 0, 1};
  if (sms < 1 || n_items <= sms) return sp;
  const long long tail = n_items % sms;
  if (tail == 0) return sp;
  const long long whole = nK + KEY_SPLIT_ITEM_TILES;
  int best = 1;
  long long best_cost = whole;
  for (int s = 2; s <= max_parts && s <= KEY_SPLIT_MAX_PARTS; ++s) {
    if (nK < KEY_SPLIT_MIN_TILES * s) break;
    const long long rounds = (tail * s + sms - 1) / sms;
    const long long cost = rounds * ((nK + s - 1) / s + KEY_SPLIT_ITEM_TILES) + KEY_SPLIT_MERGE_TILES;
    if (cost < best_cost) {
      best = s;
      best_cost = cost;
    }
  }
  if (best == 1 || 100 * best_cost > 85 * whole) return sp;
  sp.n_whole = n_items - tail;
  sp.n_tail = tail;
  sp.n_parts = best;
  return sp;
}

// The split of a launch (fixed length, not causal) on the current device, and the workspace it
// needs: per cut range, 128 * (query tiles per CTA) rows of D fp32 partial outputs, then one fp32
// lse per row.  0 bytes (and n_parts = 1) when the launch runs unsplit.
struct KeySplit {
  SplitPlan plan{0, 0, 1};
  size_t o_bytes = 0, l_bytes = 0;
  size_t bytes() const { return o_bytes + l_bytes; }
};

int plan_key_split(long long n_items, int nK, int D, int causal, KeySplit* ks) {
  *ks = KeySplit{};
  ks->plan.n_whole = n_items;
  const int max_parts = g_key_split_max.load();
  if (causal || max_parts < 2) return ATTN_OK;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
  const SplitPlan sp = key_split_plan(n_items, sms, nK, max_parts);
  if (sp.n_parts < 2) return ATTN_OK;
  if (sp.n_whole > 0x7fffffffll || sp.n_tail > 0x7fffffffll)
    return fail(ATTN_ERR_INVALID_ARG, "too many query blocks");
  ks->plan = sp;
  const size_t rows = 128ull * attn_q_tiles(D) * sp.n_tail * sp.n_parts;
  ks->o_bytes = rows * D * 4;
  ks->l_bytes = rows * 4;
  return ATTN_OK;
}

// The split parameters of a launch with the caller's workspace (nullptr: unsplit).  A
// workspace smaller than the plan needs is an error, never a silent fallback: the same
// arguments always give the same launches.
int key_split_params(const AttnParams& p, int D, int causal, void* ws, size_t ws_bytes, SplitParams* out,
                     bool* split) {
  *split = false;
  if (ws == nullptr) return ATTN_OK;
  KeySplit ks;
  int rc = plan_key_split(1ll * p.nQB * p.H * p.B, p.nK, D, causal, &ks);
  if (rc != ATTN_OK) return rc;
  if (ks.plan.n_parts < 2) return ATTN_OK;
  if (ws_bytes < ks.bytes())
    return fail(ATTN_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %zu the key split needs "
                "(attn_fwd_split_workspace_bytes)", ws_bytes, ks.bytes());
  char* base = static_cast<char*>(ws);
  out->n_whole = static_cast<int>(ks.plan.n_whole);
  out->n_tail = static_cast<int>(ks.plan.n_tail);
  out->n_parts = ks.plan.n_parts;
  out->part_o = reinterpret_cast<float*>(base);
  out->part_l = reinterpret_cast<float*>(base + ks.o_bytes);
  *split = true;
  return ATTN_OK;
}

// Shape and pointer checks shared by the attention entry points.
int check_attn_args(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    int B, int H, int S, int D, int causal, float scale, int esz) {
  if (q == nullptr || k == nullptr || v == nullptr || o == nullptr)
    return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be non-null device pointers");
  if (B < 1 || H < 1 || S < 1)
    return fail(ATTN_ERR_INVALID_ARG, "B, H, S must be >= 1 (got %d, %d, %d)", B, H, S);
  if (D != 64 && D != 128 && D != 256)
    return fail(D > 0 ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_INVALID_ARG,
                "head dimension D = %d not supported (64, 128, 256)", D);
  if (causal != 0 && causal != 1) return fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (!std::isfinite(scale) || scale < 0.f)
    return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and >= 0 (0 selects 1/sqrt(D))");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return fail(ATTN_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  const unsigned long long n = 1ull * B * S * H * D;
  if (n > (1ull << 40) / 2)
    return fail(ATTN_ERR_INVALID_ARG, "tensor too large (%llu elements)", n);
  const unsigned long long rows_per_cta = 128ull * attn_q_tiles(D);
  const unsigned long long grid = 1ull * ((S + rows_per_cta - 1) / rows_per_cta) * H * B;
  if (grid > 0x7fffffffull) return fail(ATTN_ERR_INVALID_ARG, "too many query blocks");
  const size_t in_bytes = n * esz, out_bytes = n * 2;
  if (overlap(o, out_bytes, q, in_bytes) || overlap(o, out_bytes, k, in_bytes) ||
      overlap(o, out_bytes, v, in_bytes))
    return fail(ATTN_ERR_INVALID_ARG, "o overlaps an input");
  if (lse != nullptr) {
    const size_t lse_bytes = 4ull * B * H * S;
    if (overlap(lse, lse_bytes, o, out_bytes) || overlap(lse, lse_bytes, q, in_bytes) ||
        overlap(lse, lse_bytes, k, in_bytes) || overlap(lse, lse_bytes, v, in_bytes))
      return fail(ATTN_ERR_INVALID_ARG, "lse overlaps another tensor");
  }
  return ATTN_OK;
}

template <bool FP8>
int dispatch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
             const AttnParams& p, int D, int causal, cudaStream_t st, const SplitParams* sp) {
  cudaError_t e = cudaErrorInvalidValue;
  switch (D * 2 + causal) {
    case 64 * 2 + 0: e = launch_attn<64, FP8, false>(tq, tk, tv, to, p, st, sp); break;
    case 64 * 2 + 1: e = launch_attn<64, FP8, true>(tq, tk, tv, to, p, st, nullptr); break;
    case 128 * 2 + 0: e = launch_attn<128, FP8, false>(tq, tk, tv, to, p, st, sp); break;
    case 128 * 2 + 1: e = launch_attn<128, FP8, true>(tq, tk, tv, to, p, st, nullptr); break;
    case 256 * 2 + 0: e = launch_attn<256, FP8, false>(tq, tk, tv, to, p, st, sp); break;
    case 256 * 2 + 1: e = launch_attn<256, FP8, true>(tq, tk, tv, to, p, st, nullptr); break;
    default: break;
  }
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "attention launch failed: %s", cudaGetErrorString(e));
  return ok();
}

int run_attn(const void* q, const void* k, const void* v, const float* qs, const float* ks,
             const float* vs, void* o, float* lse, int B, int H, int S, int D, int causal,
             float scale, bool fp8, void* stream) {
  int rc = check_attn_args(q, k, v, o, lse, B, H, S, D, causal, scale, fp8 ? 1 : 2);
  if (rc != ATTN_OK) return rc;
  int* err = nullptr;
  if ((rc = err_words(&err)) != ATTN_OK) return rc;
  CUtensorMap tq, tk, tv;
  if ((rc = make_qkv_map(&tq, q, B, S, H, D, fp8)) != ATTN_OK) return rc;
  if ((rc = make_qkv_map(&tk, k, B, S, H, D, fp8)) != ATTN_OK) return rc;
  if ((rc = make_qkv_map(&tv, v, B, S, H, D, fp8)) != ATTN_OK) return rc;
  CUtensorMap to;
  if ((rc = make_o_map(&to, o, B, S, H, D)) != ATTN_OK) return rc;
  AttnParams p{};
  p.B = B;
  p.H = H;
  p.S = S;
  const int rows_per_cta = 128 * attn_q_tiles(D);
  p.nQB = (S + rows_per_cta - 1) / rows_per_cta;
  p.nK = (S + 127) / 128;
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(D));
  p.c_log2 = sc * 1.4426950408889634f;
  p.o = o;
  p.lse = lse;
  p.q_scale = qs;
  p.k_scale = ks;
  p.v_scale = vs;
  p.spin_limit = spin_limit();
  p.err_word = err;
  p.err_info = err + 1;
  p.kv_group = 1;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return fp8 ? dispatch<true>(tq, tk, tv, to, p, D, causal, st, nullptr)
             : dispatch<false>(tq, tk, tv, to, p, D, causal, st, nullptr);
}

template <bool FP8, bool CAUSAL>
cudaError_t launch_varlen(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const AttnParams& p, int D, cudaStream_t st) {
  // the packed-batch kernels store O from registers: the O map is not read
  return D == 64    ? launch_attn<64, FP8, CAUSAL, true>(tq, tk, tv, tq, p, st, nullptr)
         : D == 128 ? launch_attn<128, FP8, CAUSAL, true>(tq, tk, tv, tq, p, st, nullptr)
                    : launch_attn<256, FP8, CAUSAL, true>(tq, tk, tv, tq, p, st, nullptr);
}

// Scale entries per head of a packed batch's block scales.
long long varlen_scale_blocks(long long total, long long n_seq) { return total / 128 + n_seq + 1; }

// One thread waits on a barrier that nothing arrives at; the bounded wait records a timeout.
__global__ void selftest_wait_kernel(long long limit, int* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtl ctl{limit, &abort_flag, err, err + 1};
    (void)wait_bounded(smem_u32(&bar), 0, ctl, 99);
  }
  __syncthreads();
}

int run_quant(const void* x, const float* rope_cs, int n_pos, void* out, float* scale, const float* signs,
              int B, int H, int S, int D, void* stream, const int* cu_seqlens = nullptr, int n_seq = 0) {
  if (x == nullptr || out == nullptr || scale == nullptr)
    return fail(ATTN_ERR_INVALID_ARG, "x, out and scale must be non-null device pointers");
  if (B < 1 || H < 1 || S < 1)
    return fail(ATTN_ERR_INVALID_ARG, "B, H, S must be >= 1 (got %d, %d, %d)", B, H, S);
  if (D != 64 && D != 128 && D != 256)
    return fail(D > 0 ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_INVALID_ARG,
                "head dimension D = %d not supported (64, 128, 256)", D);
  if (!aligned16(x) || !aligned16(out) || (signs != nullptr && !aligned16(signs)) ||
      (rope_cs != nullptr && !aligned16(rope_cs)) || (reinterpret_cast<uintptr_t>(scale) & 3u))
    return fail(ATTN_ERR_INVALID_ARG, "x, out, signs, rope_cs must be 16-byte and scale 4-byte aligned");
  const unsigned long long n = 1ull * B * S * H * D;
  const long long nblk_ll = cu_seqlens != nullptr ? varlen_scale_blocks(S, n_seq) : (S + 127) / 128;
  if (n > (1ull << 40) / 2 || nblk_ll * H * B >= 0x7fffffffll || H > 65535 || B > 65535)
    return fail(ATTN_ERR_INVALID_ARG, "tensor too large for the grid");
  const int nblk = static_cast<int>(nblk_ll);
  if (rope_cs != nullptr && cu_seqlens == nullptr && n_pos < 128 * nblk)
    return fail(ATTN_ERR_INVALID_ARG,
                "the rotary table needs rows for every position of the last 128-token block: "
                "n_pos = %d < %d", n_pos, 128 * nblk);
  const size_t sbytes = 4ull * B * H * nblk;
  if (overlap(out, n, x, 2 * n) || overlap(scale, sbytes, x, 2 * n) || overlap(scale, sbytes, out, n))
    return fail(ATTN_ERR_INVALID_ARG, "outputs overlap the input or each other");
  if (cu_seqlens != nullptr &&
      (overlap(out, n, cu_seqlens, 4ull * (n_seq + 1)) || overlap(scale, sbytes, cu_seqlens, 4ull * (n_seq + 1))))
    return fail(ATTN_ERR_INVALID_ARG, "outputs overlap cu_seqlens");
  if (rope_cs != nullptr) {
    const size_t tbytes = 4ull * n_pos * D;
    if (overlap(out, n, rope_cs, tbytes) || overlap(scale, sbytes, rope_cs, tbytes))
      return fail(ATTN_ERR_INVALID_ARG, "outputs overlap the rotary table");
  }
  int* err = nullptr;
  int rc = err_words(&err);
  if (rc != ATTN_OK) return rc;
  QuantMaps m;
  if ((rc = make_qkv_map(&m.x[0], x, B, S, H, D, false)) != ATTN_OK) return rc;
  // the quantiser stores its codes one warp's rows at a time: 32 rows, 16 at D = 256
  if ((rc = make_qkv_map(&m.out[0], out, B, S, H, D, true, D == 256 ? 16 : 32)) != ATTN_OK) return rc;
  QuantParams p{B, H, S, nblk, out, scale, signs, rope_cs, spin_limit(), err, err + 1, cu_seqlens, n_seq, n_pos};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = D == 64    ? launch_hadamard_quant<64>(m, p, st)
                  : D == 128 ? launch_hadamard_quant<128>(m, p, st)
                             : launch_hadamard_quant<256>(m, p, st);
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "quantiser launch failed: %s", cudaGetErrorString(e));
  return ok();
}

// Q, K and V in one quantiser launch: Q and K rotated (when signs is given), V not.
int run_quant_qkv(const void* const x[3], void* const out[3], float* const scale[3], const float* signs, int B,
                  int H, int S, int D, void* stream) {
  for (int t = 0; t < 3; ++t)
    if (x[t] == nullptr || out[t] == nullptr || scale[t] == nullptr)
      return fail(ATTN_ERR_INVALID_ARG, "q, k, v, their codes and their scales must be non-null device pointers");
  if (B < 1 || H < 1 || S < 1)
    return fail(ATTN_ERR_INVALID_ARG, "B, H, S must be >= 1 (got %d, %d, %d)", B, H, S);
  if (D != 64 && D != 128 && D != 256)
    return fail(D > 0 ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_INVALID_ARG,
                "head dimension D = %d not supported (64, 128, 256)", D);
  for (int t = 0; t < 3; ++t)
    if (!aligned16(x[t]) || !aligned16(out[t]) || (reinterpret_cast<uintptr_t>(scale[t]) & 3u))
      return fail(ATTN_ERR_INVALID_ARG, "inputs and codes must be 16-byte and scales 4-byte aligned");
  if (signs != nullptr && !aligned16(signs)) return fail(ATTN_ERR_INVALID_ARG, "signs must be 16-byte aligned");
  const unsigned long long n = 1ull * B * S * H * D;
  const long long nblk_ll = (S + 127) / 128;
  if (n > (1ull << 40) / 2 || 3 * nblk_ll * H * B >= 0x7fffffffll || H > 65535 || B > 65535)
    return fail(ATTN_ERR_INVALID_ARG, "tensors too large for the grid");
  const int nblk = static_cast<int>(nblk_ll);
  const size_t sbytes = 4ull * B * H * nblk;
  // the six outputs overlap neither each other nor the three inputs
  const void* obuf[6] = {out[0], out[1], out[2], scale[0], scale[1], scale[2]};
  const size_t olen[6] = {n, n, n, sbytes, sbytes, sbytes};
  for (int i = 0; i < 6; ++i) {
    for (int t = 0; t < 3; ++t)
      if (overlap(obuf[i], olen[i], x[t], 2 * n)) return fail(ATTN_ERR_INVALID_ARG, "outputs overlap an input");
    for (int j = i + 1; j < 6; ++j)
      if (overlap(obuf[i], olen[i], obuf[j], olen[j])) return fail(ATTN_ERR_INVALID_ARG, "outputs overlap each other");
  }
  int* err = nullptr;
  int rc = err_words(&err);
  if (rc != ATTN_OK) return rc;
  QuantMaps m;
  for (int t = 0; t < 3; ++t) {
    if ((rc = make_qkv_map(&m.x[t], x[t], B, S, H, D, false)) != ATTN_OK) return rc;
    if ((rc = make_qkv_map(&m.out[t], out[t], B, S, H, D, true, D == 256 ? 16 : 32)) != ATTN_OK) return rc;
  }
  QuantParams p{B, H, S, nblk, out[0], scale[0], signs, nullptr, spin_limit(), err, err + 1, nullptr, 0, 0};
  p.n_tensors = 3;
  p.rot_tensors = signs != nullptr ? 2 : 0;
  p.scale1 = scale[1];
  p.scale2 = scale[2];
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = D == 64    ? launch_hadamard_quant<64>(m, p, st)
                  : D == 128 ? launch_hadamard_quant<128>(m, p, st)
                             : launch_hadamard_quant<256>(m, p, st);
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "quantiser launch failed: %s", cudaGetErrorString(e));
  return ok();
}

// Key splits for decoding.  Each CTA pays a fixed start-up (barriers, Tensor Memory, the query
// tile, filling the K/V ring, the epilogue) worth about three 128-key tiles, then streams its
// tiles at the SM's share of HBM bandwidth; the split count minimises
// waves * (3 + tiles per split), waves = ceil(B * Hkv * splits / SMs), fewest splits on ties.
void decode_plan(int B, int Hkv, int Sk, int* n_split, int* tps) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0) sms = n;
  }
  const long long base = 1ll * B * Hkv;
  const int nk = (Sk + 127) / 128;
  int best_t = nk;
  long long best = -1;
  for (int n = 1; n <= 64 && n <= nk; ++n) {
    const int t = (nk + n - 1) / n;
    const int eff_n = (nk + t - 1) / t;       // splits that actually hold tiles
    const long long waves = (base * eff_n + sms - 1) / sms;
    const long long cost = waves * (3 + t);
    if (best < 0 || cost < best) {
      best = cost;
      best_t = t;
    }
  }
  *tps = best_t;
  *n_split = (nk + best_t - 1) / best_t;
}

int make_q_group_map(CUtensorMap* m, const void* q, int B, int Sq, int Hkv, int G, int D, bool fp8) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  const int esz = fp8 ? 1 : 2;
  const int panel_row = D * esz >= 128 ? 128 : D * esz;
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(G), static_cast<cuuint64_t>(Hkv),
                              static_cast<cuuint64_t>(Sq), static_cast<cuuint64_t>(B)};
  const cuuint64_t row = static_cast<cuuint64_t>(D) * esz;
  const cuuint64_t strides[4] = {row, row * G, row * G * Hkv, row * G * Hkv * Sq};
  const cuuint32_t box[5] = {static_cast<cuuint32_t>(panel_row / esz), static_cast<cuuint32_t>(G), 1,
                             static_cast<cuuint32_t>(Sq), 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5,
                         const_cast<void*>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         panel_row == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                         l2_promotion(D * esz), CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled (grouped Q) failed (%d)", int(r));
  return ATTN_OK;
}

// Pointer / shape checks of the grouped-head entry points: q and o carry Hq heads over Sq
// tokens, k and v Hkv heads over Sk tokens.
int check_gqa_args(const void* q, const void* k, const void* v, const void* o, const float* lse, int B, int Hq,
                   int Hkv, int Sq, int Sk, int D, int causal, float scale, bool d256_ok, int esz = 2) {
  if (Hkv < 1 || Hq < 1 || Hq % Hkv != 0)
    return fail(ATTN_ERR_INVALID_ARG, "Hq (%d) must be a positive multiple of Hkv (%d)", Hq, Hkv);
  if (Sk < 1 || Sq < 1 || Sq > Sk) return fail(ATTN_ERR_INVALID_ARG, "need 1 <= Sq <= Sk (got %d, %d)", Sq, Sk);
  if (D == 256 && !d256_ok) return fail(ATTN_ERR_UNSUPPORTED, "D = 256 is not supported here (64, 128)");
  int rc = check_attn_args(q, q, q, o, lse, B, Hq, Sq, D, causal, scale, esz);   // q, o, lse
  if (rc != ATTN_OK) return rc;
  if (k == nullptr || v == nullptr || !aligned16(k) || !aligned16(v))
    return fail(ATTN_ERR_INVALID_ARG, "k and v must be non-null, 16-byte aligned device pointers");
  const size_t kvb = 1ull * esz * B * Sk * Hkv * D, ob = 2ull * B * Sq * Hq * D, lb = 4ull * B * Hq * Sq;
  if (overlap(o, ob, k, kvb) || overlap(o, ob, v, kvb) ||
      (lse != nullptr && (overlap(lse, lb, k, kvb) || overlap(lse, lb, v, kvb))))
    return fail(ATTN_ERR_INVALID_ARG, "an output overlaps k or v");
  return ATTN_OK;
}

// The backward pass: H query heads over Hkv key/value heads (Hkv = H: plain multi-head).
int run_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
            void* dq, void* dk, void* dv, float* workspace, size_t workspace_bytes, int B, int H, int Hkv, int S,
            int D, int causal, float scale, void* stream) {
  if (o == nullptr || dout == nullptr || lse == nullptr || dq == nullptr || dk == nullptr || dv == nullptr ||
      workspace == nullptr)
    return fail(ATTN_ERR_INVALID_ARG, "o, dout, lse, dq, dk, dv and workspace must be non-null device pointers");
  if (D == 256) return fail(ATTN_ERR_UNSUPPORTED, "the backward pass supports D = 64 and 128 (got 256)");
  int rc = check_gqa_args(q, k, v, dq, nullptr, B, H, Hkv, S, S, D, causal, scale, false, 2);
  if (rc != ATTN_OK) return rc;
  if (!aligned16(o) || !aligned16(dout) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(ATTN_ERR_INVALID_ARG, "tensors and workspace must be 16-byte aligned (lse 4-byte)");
  const size_t need = attn_bwd_workspace_bytes(B, H, S);
  if (workspace_bytes < need)
    return fail(ATTN_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %zu needed", workspace_bytes, need);
  const size_t n = 2ull * B * S * H * D, nkv = 2ull * B * S * Hkv * D, nl = 4ull * B * H * S;
  const void* ins[6] = {q, k, v, o, dout, lse};
  const size_t in_bytes[6] = {n, nkv, nkv, n, n, nl};
  void* outs[4] = {dq, dk, dv, workspace};
  const size_t out_bytes[4] = {n, nkv, nkv, need};
  for (int a = 0; a < 4; ++a) {
    for (int i = 0; i < 6; ++i)
      if (overlap(outs[a], out_bytes[a], ins[i], in_bytes[i]))
        return fail(ATTN_ERR_INVALID_ARG, "an output or the workspace overlaps an input");
    for (int c = a + 1; c < 4; ++c)
      if (overlap(outs[a], out_bytes[a], outs[c], out_bytes[c]))
        return fail(ATTN_ERR_INVALID_ARG, "outputs overlap each other or the workspace");
  }
  int* err = nullptr;
  if ((rc = err_words(&err)) != ATTN_OK) return rc;
  CUtensorMap maps[4];
  const void* srcs[4] = {q, k, v, dout};
  for (int i = 0; i < 4; ++i)
    if ((rc = make_qkv_map(&maps[i], srcs[i], B, S, (i == 1 || i == 2) ? Hkv : H, D, false)) != ATTN_OK) return rc;
  BwdParams p{};
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.S = S;
  p.Sp = (S + 127) / 128 * 128;
  p.scale = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(D));
  p.c_log2 = p.scale * 1.4426950408889634f;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.ws = workspace;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.spin_limit = spin_limit();
  p.err_word = err;
  p.err_info = err + 1;
  const cudaError_t e = launch_attn_bwd(maps, p, D, causal != 0, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "backward launch failed: %s", cudaGetErrorString(e));
  return ok();
}

// Grouped-query prefill: bf16 inputs (qs = ks = vs = nullptr) or E4M3 codes with block scales
// (q_scale [B, Hq, nK], k_scale and v_scale [B, Hkv, nK]).
int run_gqa(const void* q, const void* k, const void* v, const float* qs, const float* ks, const float* vs, void* o,
            float* lse, int B, int Hq, int Hkv, int S, int D, int causal, float scale, bool fp8, void* stream,
            void* ws = nullptr, size_t ws_bytes = 0) {
  int rc = check_gqa_args(q, k, v, o, lse, B, Hq, Hkv, S, S, D, causal, scale, true, fp8 ? 1 : 2);
  if (rc != ATTN_OK) return rc;
  if (ws != nullptr) {
    if (!aligned16(ws)) return fail(ATTN_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    const size_t nq = 1ull * B * S * Hq * D, nkv = 1ull * B * S * Hkv * D, esz = fp8 ? 1 : 2;
    if (overlap(ws, ws_bytes, q, nq * esz) || overlap(ws, ws_bytes, k, nkv * esz) ||
        overlap(ws, ws_bytes, v, nkv * esz) || overlap(ws, ws_bytes, o, nq * 2) ||
        (lse != nullptr && overlap(ws, ws_bytes, lse, 4ull * B * Hq * S)))
      return fail(ATTN_ERR_INVALID_ARG, "workspace overlaps an input or output");
  }
  int* err = nullptr;
  if ((rc = err_words(&err)) != ATTN_OK) return rc;
  CUtensorMap tq, tk, tv;
  if ((rc = make_qkv_map(&tq, q, B, S, Hq, D, fp8)) != ATTN_OK) return rc;
  if ((rc = make_qkv_map(&tk, k, B, S, Hkv, D, fp8)) != ATTN_OK) return rc;
  if ((rc = make_qkv_map(&tv, v, B, S, Hkv, D, fp8)) != ATTN_OK) return rc;
  CUtensorMap to;
  if ((rc = make_o_map(&to, o, B, S, Hq, D)) != ATTN_OK) return rc;
  AttnParams p{};
  p.B = B;
  p.H = Hq;
  p.S = S;
  const int rows_per_cta = 128 * attn_q_tiles(D);
  p.nQB = (S + rows_per_cta - 1) / rows_per_cta;
  p.nK = (S + 127) / 128;
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(D));
  p.c_log2 = sc * 1.4426950408889634f;
  p.o = o;
  p.lse = lse;
  p.q_scale = qs;
  p.k_scale = ks;
  p.v_scale = vs;
  p.spin_limit = spin_limit();
  p.err_word = err;
  p.err_info = err + 1;
  p.kv_group = Hq / Hkv;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  SplitParams sp{};
  bool split = false;
  if ((rc = key_split_params(p, D, causal, ws, ws_bytes, &sp, &split)) != ATTN_OK) return rc;
  return fp8 ? dispatch<true>(tq, tk, tv, to, p, D, causal, st, split ? &sp : nullptr)
             : dispatch<false>(tq, tk, tv, to, p, D, causal, st, split ? &sp : nullptr);
}

}  // namespace

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int S, int D, int causal, float scale, int dtype, void* stream) {
  if (dtype != ATTN_BF16 && dtype != ATTN_FP8_E4M3)
    return fail(ATTN_ERR_INVALID_ARG, "dtype must be ATTN_BF16 (0) or ATTN_FP8_E4M3 (1)");
  return run_attn(q, k, v, nullptr, nullptr, nullptr, o, lse, B, H, S, D, causal, scale,
                  dtype == ATTN_FP8_E4M3, stream);
}

int attn_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* q_scale,
                 const float* k_scale, const float* v_scale, void* o, float* lse, int B, int H,
                 int S, int D, int causal, float scale, void* stream) {
  if (q_scale == nullptr || k_scale == nullptr || v_scale == nullptr)
    return fail(ATTN_ERR_INVALID_ARG, "q_scale, k_scale and v_scale must be non-null");
  if ((reinterpret_cast<uintptr_t>(q_scale) | reinterpret_cast<uintptr_t>(k_scale) |
       reinterpret_cast<uintptr_t>(v_scale)) & 3u)
    return fail(ATTN_ERR_INVALID_ARG, "scale arrays must be 4-byte aligned");
  return run_attn(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, B, H, S, D, causal, scale,
                  true, stream);
}

int hadamard_rotate_quant_fp8(const void* x, void* out, float* scale, const float* signs, int B,
                              int H, int S, int D, void* stream) {
  return run_quant(x, nullptr, 0, out, scale, signs, B, H, S, D, stream);
}

int hadamard_rotate_quant_fp8_qkv(const void* q, const void* k, const void* v, void* q8, void* k8, void* v8,
                                  float* q_scale, float* k_scale, float* v_scale, const float* signs, int B,
                                  int H, int S, int D, void* stream) {
  const void* x[3] = {q, k, v};
  void* out[3] = {q8, k8, v8};
  float* scale[3] = {q_scale, k_scale, v_scale};
  return run_quant_qkv(x, out, scale, signs, B, H, S, D, stream);
}

int rope_hadamard_rotate_quant_fp8(const void* x, const float* rope_cs, int n_pos, void* out, float* scale,
                                   const float* signs, int B, int H, int S, int D, void* stream) {
  if (rope_cs == nullptr) return fail(ATTN_ERR_INVALID_ARG, "rope_cs must be a non-null device pointer");
  return run_quant(x, rope_cs, n_pos, out, scale, signs, B, H, S, D, stream);
}

int rope_cos_sin_table(float* cs, int n_pos, int D, double base, void* stream) {
  if (cs == nullptr) return fail(ATTN_ERR_INVALID_ARG, "cs must be a non-null device pointer");
  if (n_pos < 1 || n_pos > (1 << 26))
    return fail(ATTN_ERR_INVALID_ARG, "n_pos must be in [1, 2^26] (got %d)", n_pos);
  if (D < 2 || D % 2 != 0 || D > 4096)
    return fail(ATTN_ERR_INVALID_ARG, "D must be even and in [2, 4096] (got %d)", D);
  if (!(base > 0.0) || !std::isfinite(base))
    return fail(ATTN_ERR_INVALID_ARG, "base must be finite and > 0");
  if (reinterpret_cast<uintptr_t>(cs) & 7u) return fail(ATTN_ERR_INVALID_ARG, "cs must be 8-byte aligned");
  cudaError_t e = launch_rope_table(cs, n_pos, D, base, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "rotary table launch failed: %s", cudaGetErrorString(e));
  return ok();
}

}  // extern "C"

namespace {

// Packed variable-length batches: bf16 inputs (qs = ks = vs = nullptr) or E4M3 codes with the
// block scales of hadamard_rotate_quant_fp8_varlen ([H, varlen_scale_blocks(total, n_seq)]).
int run_varlen(const void* q, const void* k, const void* v, const float* qs, const float* ks, const float* vs,
               void* o, float* lse, const int* cu_seqlens, int n_seq, int total, int max_seqlen, int H, int D,
               int causal, float scale, bool fp8, void* stream) {
  if (cu_seqlens == nullptr || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
    return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens must be a non-null, 4-byte aligned device pointer");
  if (n_seq < 1 || n_seq > VARLEN_MAX_SEQ)
    return fail(ATTN_ERR_INVALID_ARG, "n_seq must be in [1, %d] (got %d)", VARLEN_MAX_SEQ, n_seq);
  int rc = check_attn_args(q, k, v, o, lse, 1, H, total, D, causal, scale, fp8 ? 1 : 2);
  if (rc != ATTN_OK) return rc;
  const int rows_per_cta = 128 * attn_q_tiles(D);
  if (max_seqlen < 1)
    return fail(ATTN_ERR_INVALID_ARG, "max_seqlen must be >= 1 (got %d)", max_seqlen);
  if (max_seqlen > VARLEN_MAX_LEVELS * rows_per_cta)
    return fail(ATTN_ERR_UNSUPPORTED, "max_seqlen %d above the limit %d for D = %d", max_seqlen,
                VARLEN_MAX_LEVELS * rows_per_cta, D);
  if ((static_cast<long long>(total) / 128 + n_seq) * H >= (1ll << 31))
    return fail(ATTN_ERR_INVALID_ARG, "too many work items (total / 128 + n_seq) * H");
  const size_t lse_bytes = lse != nullptr ? 4ull * H * total : 0;
  if (lse != nullptr && overlap(cu_seqlens, 4ull * (n_seq + 1), lse, lse_bytes))
    return fail(ATTN_ERR_INVALID_ARG, "lse overlaps cu_seqlens");
  if (overlap(cu_seqlens, 4ull * (n_seq + 1), o, 2ull * total * H * D))
    return fail(ATTN_ERR_INVALID_ARG, "o overlaps cu_seqlens");
  int* err = nullptr;
  if ((rc = err_words(&err)) != ATTN_OK) return rc;
  CUtensorMap tq, tk, tv;
  if ((rc = make_qkv_map(&tq, q, 1, total, H, D, fp8)) != ATTN_OK) return rc;
  if ((rc = make_qkv_map(&tk, k, 1, total, H, D, fp8)) != ATTN_OK) return rc;
  if ((rc = make_qkv_map(&tv, v, 1, total, H, D, fp8)) != ATTN_OK) return rc;
  AttnParams p{};
  p.B = 1;
  p.H = H;
  p.S = total;
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(D));
  p.c_log2 = sc * 1.4426950408889634f;
  p.o = o;
  p.lse = lse;
  p.spin_limit = spin_limit();
  p.err_word = err;
  p.err_info = err + 1;
  p.cu_seqlens = cu_seqlens;
  p.n_seq = n_seq;
  p.kv_group = 1;
  p.max_seqlen = max_seqlen;
  p.n_levels = (max_seqlen + rows_per_cta - 1) / rows_per_cta;
  p.q_scale = qs;
  p.k_scale = ks;
  p.v_scale = vs;
  p.scale_stride = static_cast<int>(varlen_scale_blocks(total, n_seq));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (fp8) e = causal ? launch_varlen<true, true>(tq, tk, tv, p, D, st) : launch_varlen<true, false>(tq, tk, tv, p, D, st);
  else e = causal ? launch_varlen<false, true>(tq, tk, tv, p, D, st) : launch_varlen<false, false>(tq, tk, tv, p, D, st);
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
  return ok();
}

}  // namespace

extern "C" {

int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens,
                    int n_seq, int total, int max_seqlen, int H, int D, int causal, float scale, void* stream) {
  return run_varlen(q, k, v, nullptr, nullptr, nullptr, o, lse, cu_seqlens, n_seq, total, max_seqlen, H, D, causal,
                    scale, false, stream);
}

int attn_fwd_varlen_fp8(const void* q8, const void* k8, const void* v8, const float* q_scale, const float* k_scale,
                        const float* v_scale, void* o, float* lse, const int* cu_seqlens, int n_seq, int total,
                        int max_seqlen, int H, int D, int causal, float scale, void* stream) {
  if (q_scale == nullptr || k_scale == nullptr || v_scale == nullptr)
    return fail(ATTN_ERR_INVALID_ARG, "q_scale, k_scale and v_scale must be non-null");
  if ((reinterpret_cast<uintptr_t>(q_scale) | reinterpret_cast<uintptr_t>(k_scale) |
       reinterpret_cast<uintptr_t>(v_scale)) & 3u)
    return fail(ATTN_ERR_INVALID_ARG, "scale arrays must be 4-byte aligned");
  return run_varlen(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, cu_seqlens, n_seq, total, max_seqlen, H, D,
                    causal, scale, true, stream);
}

int attn_varlen_scale_blocks(int total, int n_seq) {
  if (total < 0 || n_seq < 0) return 0;
  const long long nb = varlen_scale_blocks(total, n_seq);
  return nb > 0x7fffffffll ? 0 : static_cast<int>(nb);
}

int hadamard_rotate_quant_fp8_varlen(const void* x, void* out, float* scale, const float* signs,
                                     const int* cu_seqlens, int n_seq, int total, int H, int D, void* stream) {
  if (cu_seqlens == nullptr || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
    return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens must be a non-null, 4-byte aligned device pointer");
  if (n_seq < 1 || n_seq > VARLEN_MAX_SEQ)
    return fail(ATTN_ERR_INVALID_ARG, "n_seq must be in [1, %d] (got %d)", VARLEN_MAX_SEQ, n_seq);
  return run_quant(x, nullptr, 0, out, scale, signs, 1, H, total, D, stream, cu_seqlens, n_seq);
}

int rope_hadamard_rotate_quant_fp8_varlen(const void* x, const float* rope_cs, int n_pos, void* out, float* scale,
                                          const float* signs, const int* cu_seqlens, int n_seq, int total, int H,
                                          int D, void* stream) {
  if (rope_cs == nullptr) return fail(ATTN_ERR_INVALID_ARG, "rope_cs must be a non-null device pointer");
  if (n_pos < 128)
    return fail(ATTN_ERR_INVALID_ARG, "the rotary table needs at least the 128 rows of one block (n_pos = %d)", n_pos);
  if (cu_seqlens == nullptr || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
    return fail(ATTN_ERR_INVALID_ARG, "cu_seqlens must be a non-null, 4-byte aligned device pointer");
  if (n_seq < 1 || n_seq > VARLEN_MAX_SEQ)
    return fail(ATTN_ERR_INVALID_ARG, "n_seq must be in [1, %d] (got %d)", VARLEN_MAX_SEQ, n_seq);
  return run_quant(x, rope_cs, n_pos, out, scale, signs, 1, H, total, D, stream, cu_seqlens, n_seq);
}

size_t attn_bwd_workspace_bytes(int B, int H, int S) {
  if (B < 1 || H < 1 || S < 1) return 0;
  return 8ull * B * H * ((static_cast<size_t>(S) + 127) / 128 * 128);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
             void* dq, void* dk, void* dv, float* workspace, size_t workspace_bytes, int B, int H, int S, int D,
             int causal, float scale, void* stream) {
  return run_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, H, S, D, causal, scale, stream);
}

int attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 void* dq, void* dk, void* dv, float* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                 int S, int D, int causal, float scale, void* stream) {
  if (Hkv < 1 || Hq < 1 || Hq % Hkv != 0)
    return fail(ATTN_ERR_INVALID_ARG, "Hq (%d) must be a positive multiple of Hkv (%d)", Hq, Hkv);
  return run_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, S, D, causal, scale,
                 stream);
}

int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, int B, int H, int S, int D, int causal,
                     float scale, void* stream) {
  const size_t need = attn_bwd_workspace_bytes(B, H, S);
  if (need == 0) return fail(ATTN_ERR_INVALID_ARG, "B, H, S must be >= 1 (got %d, %d, %d)", B, H, S);
  if (need > NOALLOC_BWD_SCRATCH_BYTES)
    return fail(ATTN_ERR_INVALID_ARG,
                "this problem needs %zu bytes of backward workspace but the built-in scratch holds %zu "
                "(B * H * S, with S rounded up to 128, must be <= %zu); call attn_bwd with a workspace instead",
                need, NOALLOC_BWD_SCRATCH_BYTES, NOALLOC_BWD_SCRATCH_BYTES / 8);
  float* ws = nullptr;
  const cudaError_t e = noalloc_bwd_scratch(&ws);
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "built-in scratch address: %s", cudaGetErrorString(e));
  return attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, ws, NOALLOC_BWD_SCRATCH_BYTES, B, H, S, D, causal, scale,
                  stream);
}

int attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int S,
                 int D, int causal, float scale, void* stream) {
  return run_gqa(q, k, v, nullptr, nullptr, nullptr, o, lse, B, Hq, Hkv, S, D, causal, scale, false, stream);
}

int attn_fwd_gqa_fp8(const void* q8, const void* k8, const void* v8, const float* q_scale, const float* k_scale,
                     const float* v_scale, void* o, float* lse, int B, int Hq, int Hkv, int S, int D, int causal,
                     float scale, void* stream) {
  if (q_scale == nullptr || k_scale == nullptr || v_scale == nullptr)
    return fail(ATTN_ERR_INVALID_ARG, "q_scale, k_scale and v_scale must be non-null");
  if ((reinterpret_cast<uintptr_t>(q_scale) | reinterpret_cast<uintptr_t>(k_scale) |
       reinterpret_cast<uintptr_t>(v_scale)) & 3u)
    return fail(ATTN_ERR_INVALID_ARG, "scale arrays must be 4-byte aligned");
  return run_gqa(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, B, Hq, Hkv, S, D, causal, scale, true, stream);
}

size_t attn_decode_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Sk < 1 || D < 1) return 0;
  int n_split = 1, tps = 1;
  decode_plan(B, Hkv, Sk, &n_split, &tps);
  if (n_split == 1) return 0;
  return 4ull * n_split * B * Hq * Sq * (static_cast<size_t>(D) + 1);
}

}  // extern "C"

namespace {

// The decoding entry points: bf16 inputs (qs = ks = vs = nullptr, fp8 = false) or E4M3 codes
// with their block scales.
int run_decode(const void* q, const void* k, const void* v, const float* qs, const float* ks, const float* vs,
               void* o, float* lse, float* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int Sq,
               int Sk, int D, int causal, float scale, bool fp8, void* stream) {
  const int esz = fp8 ? 1 : 2;
  int rc = check_gqa_args(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, false, esz);
  if (rc != ATTN_OK) return rc;
  const int G = Hq / Hkv;
  if (G * Sq > 128)
    return fail(ATTN_ERR_UNSUPPORTED, "decoding packs (Hq / Hkv) * Sq = %d query rows into one 128-row tile; "
                "use attn_fwd_gqa for longer query blocks", G * Sq);
  int n_split = 1, tps = 1;
  decode_plan(B, Hkv, Sk, &n_split, &tps);
  const size_t need = n_split == 1 ? 0 : 4ull * n_split * B * Hq * Sq * (static_cast<size_t>(D) + 1);
  if (need > 0) {
    if (workspace == nullptr || workspace_bytes < need)
      return fail(ATTN_ERR_INVALID_ARG, "decoding needs a workspace of %zu bytes (attn_decode_workspace_bytes)", need);
    if (!aligned16(workspace)) return fail(ATTN_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    const size_t qb = 1ull * esz * B * Sq * Hq * D, kvb = 1ull * esz * B * Sk * Hkv * D, ob = 2ull * B * Sq * Hq * D;
    if (overlap(workspace, need, q, qb) || overlap(workspace, need, k, kvb) || overlap(workspace, need, v, kvb) ||
        overlap(workspace, need, o, ob) || (lse != nullptr && overlap(workspace, need, lse, 4ull * B * Hq * Sq)))
      return fail(ATTN_ERR_INVALID_ARG, "the workspace overlaps a tensor");
  }
  int* err = nullptr;
  if ((rc = err_words(&err)) != ATTN_OK) return rc;
  CUtensorMap tq, tk, tv;
  if ((rc = make_q_group_map(&tq, q, B, Sq, Hkv, G, D, fp8)) != ATTN_OK) return rc;
  if ((rc = make_qkv_map(&tk, k, B, Sk, Hkv, D, fp8)) != ATTN_OK) return rc;
  if ((rc = make_qkv_map(&tv, v, B, Sk, Hkv, D, fp8)) != ATTN_OK) return rc;
  DecodeParams p{};
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = G;
  p.Sq = Sq;
  p.Sk = Sk;
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(D));
  p.c_log2 = sc * 1.4426950408889634f;
  p.o = o;
  p.lse = lse;
  p.n_split = n_split;
  p.tiles_per_split = tps;
  p.rows_total = 1ll * B * Hq * Sq;
  p.ws_o = need > 0 ? workspace : nullptr;
  p.ws_l = need > 0 ? workspace + static_cast<size_t>(n_split) * p.rows_total * D : nullptr;
  p.spin_limit = spin_limit();
  p.err_word = err;
  p.err_info = err + 1;
  p.q_scale = qs;
  p.k_scale = ks;
  p.v_scale = vs;
  p.nqb = (Sq + 127) / 128;
  p.nkb = (Sk + 127) / 128;
  const cudaError_t e = launch_attn_decode(tq, tk, tv, p, D, fp8, causal != 0, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "decode launch failed: %s", cudaGetErrorString(e));
  return ok();
}

}  // namespace

extern "C" {

int attn_decode(const void* q, const void* k, const void* v, void* o, float* lse, float* workspace,
                size_t workspace_bytes, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                void* stream) {
  return run_decode(q, k, v, nullptr, nullptr, nullptr, o, lse, workspace, workspace_bytes, B, Hq, Hkv, Sq, Sk, D,
                    causal, scale, false, stream);
}

int attn_decode_fp8(const void* q8, const void* k8, const void* v8, const float* q_scale, const float* k_scale,
                    const float* v_scale, void* o, float* lse, float* workspace, size_t workspace_bytes, int B,
                    int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale, void* stream) {
  if (q_scale == nullptr || k_scale == nullptr || v_scale == nullptr)
    return fail(ATTN_ERR_INVALID_ARG, "q_scale, k_scale and v_scale must be non-null");
  if ((reinterpret_cast<uintptr_t>(q_scale) | reinterpret_cast<uintptr_t>(k_scale) |
       reinterpret_cast<uintptr_t>(v_scale)) & 3u)
    return fail(ATTN_ERR_INVALID_ARG, "scale arrays must be 4-byte aligned");
  return run_decode(q8, k8, v8, q_scale, k_scale, v_scale, o, lse, workspace, workspace_bytes, B, Hq, Hkv, Sq, Sk,
                    D, causal, scale, true, stream);
}

const char* attn_get_last_error(void) { return g_msg; }

int attn_check(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
  int* err = nullptr;
  int rc = err_words(&err);
  if (rc != ATTN_OK) return rc;
  int host[2] = {0, 0};
  e = cudaMemcpy(host, err, sizeof(host), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "error word readback: %s", cudaGetErrorString(e));
  if (host[0] != 0) {
    e = cudaMemset(err, 0, sizeof(host));
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "error word reset: %s", cudaGetErrorString(e));
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "error word reset: %s", cudaGetErrorString(e));
    if (host[0] == ATTN_ERR_INVALID_ARG)
      return fail(host[0], "a kernel rejected its device-side input (site %d: cu_seqlens must run from 0 to "
                  "total, non-decreasing, no sequence longer than max_seqlen)", host[1]);
    return fail(host[0], "a kernel's bounded wait ran out (code %d, site %d)", host[0], host[1]);
  }
  return ok();
}

void attn_set_spin_limit(long long cycles) { g_spin_limit.store(cycles > 0 ? cycles : 0); }

int attn_selftest_bounded_wait(long long spin_cycles, void* stream) {
  if (spin_cycles <= 0) return fail(ATTN_ERR_INVALID_ARG, "spin_cycles must be > 0");
  int* err = nullptr;
  int rc = err_words(&err);
  if (rc != ATTN_OK) return rc;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(spin_cycles, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
  return ok();
}

int attn_version(void) { return 120; }

void attn_set_key_split(int max_parts) {
  g_key_split_max.store(max_parts < 1 ? 1 : (max_parts > KEY_SPLIT_MAX_PARTS ? KEY_SPLIT_MAX_PARTS : max_parts));
}

int attn_key_split_plan(long long n_items, int sms, int key_tiles, int max_parts, long long* out) {
  if (out == nullptr || n_items < 0 || sms < 1 || key_tiles < 0)
    return fail(ATTN_ERR_INVALID_ARG, "need out != NULL, n_items >= 0, sms >= 1, key_tiles >= 0");
  const SplitPlan sp = key_split_plan(n_items, sms, key_tiles, max_parts);
  out[0] = sp.n_whole;
  out[1] = sp.n_tail;
  out[2] = sp.n_parts;
  return ok();
}

size_t attn_fwd_split_workspace_bytes(int B, int Hq, int S, int D, int causal) {
  if (B < 1 || Hq < 1 || S < 1 || (D != 64 && D != 128 && D != 256) || (causal != 0 && causal != 1)) return 0;
  const long long rows_per_cta = 128ll * attn_q_tiles(D);
  const long long n_items = 1ll * ((S + rows_per_cta - 1) / rows_per_cta) * Hq * B;
  KeySplit ks;
  if (plan_key_split(n_items, (S + 127) / 128, D, causal, &ks) != ATTN_OK) return 0;
  return ks.bytes();
}

int attn_fwd_split(const void* q, const void* k, const void* v, const float* q_scale, const float* k_scale,
                   const float* v_scale, void* o, float* lse, int B, int Hq, int Hkv, int S, int D, int causal,
                   float scale, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  if (dtype != ATTN_BF16 && dtype != ATTN_FP8_E4M3)
    return fail(ATTN_ERR_INVALID_ARG, "dtype must be ATTN_BF16 (0) or ATTN_FP8_E4M3 (1)");
  const int n_scales = (q_scale != nullptr) + (k_scale != nullptr) + (v_scale != nullptr);
  if (dtype == ATTN_BF16 && n_scales != 0) return fail(ATTN_ERR_INVALID_ARG, "bf16 inputs take no scales");
  if (n_scales != 0 && n_scales != 3)
    return fail(ATTN_ERR_INVALID_ARG, "give all three scale arrays or none (unit scales)");
  if ((reinterpret_cast<uintptr_t>(q_scale) | reinterpret_cast<uintptr_t>(k_scale) |
       reinterpret_cast<uintptr_t>(v_scale)) & 3u)
    return fail(ATTN_ERR_INVALID_ARG, "scale arrays must be 4-byte aligned");
  return run_gqa(q, k, v, q_scale, k_scale, v_scale, o, lse, B, Hq, Hkv, S, D, causal, scale,
                 dtype == ATTN_FP8_E4M3, stream, workspace, workspace_bytes);
}

}  // extern "C"
