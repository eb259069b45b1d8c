// attn_kernel.cuh -- fused exact-attention forward for sm_103a (tcgen05 + TMA + Tensor Memory).
//
// What it computes (hada.io FA3 summary, "Rückblick auf den FlashAttention-Ansatz" and
// "Überlappung von GEMM und Softmax"): for every query row, O = softmax(scale * q K^T) V over
// the visible keys and lse = log sum exp, reading Q, K, V once per query block and never
// writing the score matrix to device memory.  The softmax is computed tile by tile with a
// running max and running sum (softmax rescaling), which reaches the exact result.
//
// How it maps to GB300 (own design; the pages' Hopper schedule -- WGMMA warpgroups,
// ping-pong between two consumer warpgroups, intra-warpgroup overlap -- is prior art):
//
//   CTA = NT query tiles of 128 rows of one (b, h)   (NT = 2, or 1 at D = 256)
//   warps 0 .. 4*NT-1  : softmax; warp w owns query tile w/4 and Tensor-Memory lanes
//                        32*(w%4) .. +31, i.e. thread = one query row, so row max / row sum
//                        need no shuffles
//   warp 4*NT          : TMA producer: Q tiles once, then K_0, V_0, K_1, V_1, ... into a ring
//                        of NSLOT shared-memory slots (full / empty mbarriers)
//   warp 4*NT+1        : MMA issuer (one thread): S_t = Q_t K_j^T into Tensor Memory
//                        (tcgen05.mma, operands from shared memory), then O_t += P_t V_j with
//                        P_t read from Tensor Memory where the softmax warps wrote it over S_t
//
//   Issue order per key tile j: PV_0(j-1), S_0(j), PV_1(j-1), S_1(j).  While the softmax of
//   tile 0 works on S_0(j), the tensor core runs PV_1(j-1) and S_1(j), and the other way
//   round: the two query tiles alternate between the tensor pipe and the exp/ALU pipes (the
//   role the pages' ping-pong plays on Hopper), with accumulators in Tensor Memory instead
//   of registers.
//
//   Tensor Memory (512 columns x 128 lanes x 32 bit): S_t at column 128*t (P_t overwrites its
//   first 64 (bf16) or 32 (E4M3) columns), O_t at 128*NT + D*t.
//
//   The running max is only raised when a tile's max exceeds it by more than TAU = 8 (log2
//   units); otherwise the stale max is kept, numerators stay below 2^8, and O and l need no
//   rescaling.  The result is the same function (the max cancels between numerator and l);
//   the rescale of O in Tensor Memory is done by the softmax warp that owns the rows, in the
//   window where S_t(j) is ready and PV_t(j) has not been issued.
//
//   FP8 (E4M3) inputs carry one scale per (b, h, 128-token block): the logit multiplier of a
//   tile is scale*log2e*sq*sk_j; V's block scale sv_j enters as a per-tile factor
//   r_j = sv_j / max_j sv_j <= 1 folded into the exponent (p' = 2^(x - m + log2 r_j)), the row
//   sum adds sum(p') / r_j, and the epilogue multiplies by max_j sv_j / l.
//
//   Packed variable-length batches (VARLEN; hada.io FA3 summary, "Weitere Optimierungen und
//   künftige Integration", names variable-length sequences): Q, K, V are [total, H, D] with
//   sequence offsets cu_seqlens.  Every CTA copies the offsets to shared memory and sorts the
//   sequences by their number of query blocks (a stable counting sort, so every CTA derives
//   the same order), and only non-empty work items exist.  Causal: items go level by level
//   from the top query block down -- level L holds block L of every sequence longer than L
//   blocks, a prefix of the sorted order, times H heads -- so the blocks with the most keys
//   come first, as in the fixed-length order.  Otherwise: longest sequences first, and a
//   head's query blocks adjacent (its K/V then comes from L2 after the first block).  Item n
//   maps to its (sequence, head, block) by a binary search over per-level offsets.  A
//   sequence's tiles are addressed from its first token; tiles that run into the next
//   sequence are masked like the ragged tail of a fixed length, and rows past the sequence
//   are never stored.
//
//   Key-split tail (fixed length, not causal): every item is the same amount of work, so a
//   persistent grid of P CTAs runs ceil(N / P) rounds for N items and the last round is
//   partly idle.  When the host plans a split, the first n_whole = P * floor(N / P) items run
//   whole and each of the last n_tail items is cut into n_parts ranges of key tiles, so the
//   tail takes ceil(n_tail * n_parts / P) rounds of 1 / n_parts the length.  A part writes its
//   normalised partial O (fp32) and lse (log2 units) to a scratch buffer; split_merge_kernel,
//   launched next on the same stream, merges each cut row in part order (lse = log2 sum
//   2^lse_p, O = sum 2^(lse_p - lse) O_p) with a warp per row and the lanes across the
//   columns, so its reads are whole row segments.

// Every mbarrier wait is bounded (ptx.cuh, wait_bounded): a wait that runs out records
// ATTN_ERR_TIMEOUT in the device error word, raises the CTA's abort flag, and every role then
// drains its in-flight copies / MMAs and leaves through the common exit, which frees Tensor
// Memory.
#pragma once

#include <atomic>
#include <cfloat>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ea46 {

template <int D, bool FP8>
struct AttnCfg {
  static constexpr int NT = attn_q_tiles(D);
  static constexpr int ESZ = FP8 ? 1 : 2;
  static constexpr int ROW_BYTES = D * ESZ;                    // one token-head row
  static constexpr int PANEL_ROW = ROW_BYTES >= 128 ? 128 : ROW_BYTES;  // swizzle span
  static constexpr int NPANEL = ROW_BYTES / PANEL_ROW;
  static constexpr int PANEL_ELEMS = PANEL_ROW / ESZ;
  static constexpr int PANEL_BYTES = 128 * PANEL_ROW;          // 128 rows of one panel
  static constexpr int TILE_BYTES = 128 * ROW_BYTES;
  static constexpr uint32_t LAYOUT = PANEL_ROW == 128 ? 2u : 4u;   // SW128 / SW64
  static constexpr uint32_t SBO = 8 * PANEL_ROW;               // stride of 8-row groups
  // E4M3 numerators with two query tiles go through shared memory (two 128 x 128-byte buffers
  // per query tile, K-major, 128-byte swizzle) instead of over S in Tensor Memory, so the next
  // QK^T may overwrite S as soon as the softmax warps have read it
  static constexpr bool P_SMEM = FP8 && NT == 2;
  static constexpr int P_BYTES = P_SMEM ? NT * 2 * 128 * 128 : 0;
  static constexpr int SMEM_TILES_BUDGET = 200 * 1024;
  static constexpr int NSLOT_RAW = (SMEM_TILES_BUDGET - NT * TILE_BYTES - P_BYTES) / TILE_BYTES;
  static constexpr int NSLOT_CAP = P_SMEM ? 6 : 8;
  static constexpr int NSLOT = NSLOT_RAW > NSLOT_CAP ? NSLOT_CAP : NSLOT_RAW;
  // K/V ring pairs, per tile S/P/O barriers, the second Q buffer's pair, and (P_SMEM) the
  // S-read and PV-done barrier of each tile
  static constexpr int NBAR = 2 + 2 * NSLOT + 5 * NT + 1 + 2 + 2 * NT;
  static constexpr int NUM_SOFTMAX_WARPS = 4 * NT;
  // O leaves through shared memory: per softmax warp two 2 KB buffers, each 32 rows x 32
  // columns of bf16 (64-byte swizzle), stored to O by one tensor store per 32-column chunk
  static constexpr int OST_WARP_BYTES = 2 * 32 * 64;
  static constexpr int OST_BYTES = NUM_SOFTMAX_WARPS * OST_WARP_BYTES;
  // what the launch adds after the tiles and barriers: O staging, or the packed-batch tables
  static constexpr int VARLEN_TABLE_BYTES =
      ((VARLEN_MAX_SEQ + 1) + 2 * (VARLEN_MAX_LEVELS + 1) + 4) * 4 + VARLEN_MAX_SEQ * 2;
  static constexpr int EXTRA_MAX = OST_BYTES > VARLEN_TABLE_BYTES ? OST_BYTES : VARLEN_TABLE_BYTES;
  // Q tiles double-buffered where shared memory has room, so the next item's Q loads while this
  // item runs instead of after its last QK^T (at D = 128 bf16 and D = 256 it has none)
  static constexpr int QBUF =
      (2 * NT + NSLOT) * TILE_BYTES + P_BYTES + NBAR * 8 + 16 + 1024 + EXTRA_MAX <= 227 * 1024 ? 2 : 1;
  static constexpr int SMEM_BYTES_RAW = (QBUF * NT + NSLOT) * TILE_BYTES + P_BYTES + NBAR * 8 + 16;
  // Request at least ~120 KB so that one CTA (and its 512 TMEM columns) owns the SM.
  static constexpr int SMEM_BYTES =
      (SMEM_BYTES_RAW > 120 * 1024 ? SMEM_BYTES_RAW : 120 * 1024) + 1024;
  static constexpr int LOAD_WARP = NUM_SOFTMAX_WARPS;
  // MMA issuers: with P in shared memory one thread per query tile, each in a warp of its own
  // (MMA_WARP + t), so that one tile's waits never hold back the other's MMAs; otherwise one
  // thread issues both tiles' MMAs in a fixed interleave
  static constexpr int ISSUERS = P_SMEM ? NT : 1;
  static constexpr int MMA_WARP = NUM_SOFTMAX_WARPS + 1;
  static constexpr int THREADS = 32 * (NUM_SOFTMAX_WARPS + 1 + ISSUERS);
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int UMMA_K = FP8 ? 32 : 16;                 // K per MMA instruction
  static constexpr int KSTEPS_QK = ROW_BYTES / 32;             // 32 bytes of K per step
  static constexpr int STEPS_PER_PANEL = PANEL_ROW / 32;
  static constexpr int KSTEPS_PV = 128 / UMMA_K;
  static constexpr int P_COLS = 128 * ESZ / 4;                 // packed P columns (64 / 32)
  static constexpr uint32_t FMT = FP8 ? 0u : 1u;               // E4M3 / BF16
  static constexpr uint32_t IDESC_QK = instr_desc(FMT, 0, 128, 128);
  static constexpr uint32_t IDESC_PV = instr_desc(FMT, 1, 128, D);
  static_assert(128 * NT + D * NT <= 512, "Tensor Memory budget");
  static_assert(NSLOT >= 2, "need a K and a V slot");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(SMEM_BYTES + EXTRA_MAX <= 227 * 1024, "shared memory budget with O staging");
};

// Where a bounded wait gave up (reported in the error info word).
enum : int { WHERE_LOAD = 1, WHERE_MMA = 2, WHERE_SOFTMAX = 3, WHERE_DRAIN = 4 };

constexpr float TAU = 8.0f;          // log2 units a tile max may exceed the running max
constexpr float LN2 = 0.69314718055994530942f;

// Wait that ignores the abort flag: used only to drain in-flight work before exit.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, long long limit) {
  if (mbar_try_wait(bar, parity)) return;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return;
  }
}

// Epilogue of one key range of a split tail block: the warp's 32 rows of partial O
// (accumulator * inv_l, fp32) and their lse (log2 units) go to the scratch for
// split_merge_kernel (stores that bypass L1), and O_t goes back to the MMA warp.  The rows go
// through the warp's two 2 KB staging buffers, 16 columns at a time, so that each store
// instruction writes 8 rows x 64 bytes rather than 32 rows x 16 bytes.  Rows past the sequence
// (n_valid: the warp's rows that lie inside it) store nothing.  Inlined: as a call, the
// registers live across it spilled in the E4M3 kernel and slowed its key loop.
template <int D, int NT>
__device__ __forceinline__ void split_store(const SplitParams& sp, int slot, int part, int t, int row_local,
                                            bool valid, uint32_t o_addr, float inv_l, float lse2,
                                            uint32_t bar_o_empty, uint32_t ost, int n_valid) {
  constexpr int ROWS = 128 * NT;
  const uint32_t lane = lane_id();
  const size_t r = (static_cast<size_t>(slot) * sp.n_parts + part) * ROWS + 128 * t + row_local;
  // this warp's first row in the scratch; its 32 rows are consecutive there
  float* pw = sp.part_o + (r - lane) * D;
  if (lane == 0) bulk_wait_read_all();      // the item before's tensor stores have read the buffers
  __syncwarp();
#pragma unroll 1
  for (int c = 0; c < D / 32; ++c) {
    uint32_t o[32];
    tmem_ld32(o_addr + 32u * c, o);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) reg_fence(o[i]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      // 16 columns of the warp's 32 rows through buffer h (row = lane, 64 bytes, 64-byte swizzle),
      // then out with each store instruction covering 8 rows x 64 bytes
      const uint32_t buf = ost + h * (32 * 64);
#pragma unroll
      for (int v4 = 0; v4 < 4; ++v4) {
        const uint32_t addr = buf + lane * 64 + ((v4 ^ ((lane >> 1) & 3)) << 4);
        const int e = 16 * h + 4 * v4;
        st_shared_v4(addr, __float_as_uint(__uint_as_float(o[e]) * inv_l), __float_as_uint(__uint_as_float(o[e + 1]) * inv_l),
                     __float_as_uint(__uint_as_float(o[e + 2]) * inv_l), __float_as_uint(__uint_as_float(o[e + 3]) * inv_l));
      }
    }
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t buf = ost + h * (32 * 64);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = 8 * i + static_cast<int>(lane >> 2), piece = static_cast<int>(lane & 3);
        float4 f;
        // (a memory clobber: the read stays after the __syncwarp that publishes the other lanes' rows)
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(f.x), "=f"(f.y), "=f"(f.z), "=f"(f.w)
                     : "r"(buf + row * 64 + ((piece ^ ((row >> 1) & 3)) << 4))
                     : "memory");
        if (row < n_valid) __stcg(reinterpret_cast<float4*>(pw + static_cast<size_t>(row) * D + 32 * c + 16 * h + 4 * piece), f);
      }
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar_o_empty);
  if (valid) sp.part_l[r] = lse2;
}

// Merge of the split tail blocks, after the attention kernel on the same stream: one warp per
// row of a cut block, lanes across the columns.  L = log2 sum_p 2^L_p, O = sum_p 2^(L_p - L) O_p
// in part order (bf16), lse = L ln 2.
template <int D, int NT>
__global__ void __launch_bounds__(256) split_merge_kernel(const AttnParams p, const SplitParams sp) {
  constexpr int ROWS = 128 * NT;
  constexpr int CPL = D / 32;
  const long long wid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = static_cast<int>(threadIdx.x & 31);
  if (wid >= static_cast<long long>(sp.n_tail) * ROWS) return;
  const int slot = static_cast<int>(wid / ROWS), ir = static_cast<int>(wid % ROWS);
  const int id = sp.n_whole + slot;                // the cut block's item (not causal)
  const int qb = id % p.nQB, hb = id / p.nQB;
  const int h = hb % p.H, b = hb / p.H;
  const int row = qb * ROWS + ir;
  if (row >= p.S) return;
  const uint64_t drop = l2_policy_evict_first();
  const size_t r0 = static_cast<size_t>(slot) * sp.n_parts * ROWS + ir;   // part 0's row
  float lp[KEY_SPLIT_MAX_PARTS];
  float lmax = -INFINITY;
#pragma unroll
  for (int q = 0; q < KEY_SPLIT_MAX_PARTS; ++q) {
    lp[q] = q < sp.n_parts ? __ldcg(sp.part_l + r0 + static_cast<size_t>(q) * ROWS) : -INFINITY;
    lmax = fmaxf(lmax, lp[q]);
  }
  float sum = 0.f;
#pragma unroll
  for (int q = 0; q < KEY_SPLIT_MAX_PARTS; ++q) sum += q < sp.n_parts ? ex2(lp[q] - lmax) : 0.f;
  const float L = lmax + __log2f(sum);
  float x[KEY_SPLIT_MAX_PARTS][CPL];
#pragma unroll
  for (int q = 0; q < KEY_SPLIT_MAX_PARTS; ++q) {
    const float* src = sp.part_o + (r0 + static_cast<size_t>(q) * ROWS) * D + CPL * lane;
#pragma unroll
    for (int e = 0; e < CPL; e += (CPL >= 4 ? 4 : 2)) {
      if (q < sp.n_parts) {
        if constexpr (CPL >= 4) {
          const float4 v = ld_cg_v4_hint(src + e, drop);
          x[q][e] = v.x; x[q][e + 1] = v.y; x[q][e + 2] = v.z; x[q][e + 3] = v.w;
        } else {
          const float2 v = ld_cg_v2_hint(src + e, drop);
          x[q][e] = v.x; x[q][e + 1] = v.y;
        }
      } else {
#pragma unroll
        for (int f = 0; f < (CPL >= 4 ? 4 : 2); ++f) x[q][e + f] = 0.f;
      }
    }
  }
  float acc[CPL];
#pragma unroll
  for (int e = 0; e < CPL; ++e) acc[e] = 0.f;
#pragma unroll
  for (int q = 0; q < KEY_SPLIT_MAX_PARTS; ++q) {
    const float w = q < sp.n_parts ? ex2(lp[q] - L) : 0.f;
#pragma unroll
    for (int e = 0; e < CPL; ++e) acc[e] = fmaf(w, x[q][e], acc[e]);
  }
  uint32_t pk[CPL / 2];
#pragma unroll
  for (int e = 0; e < CPL / 2; ++e) pk[e] = pack_bf16x2(acc[2 * e], acc[2 * e + 1]);
  const size_t tok = static_cast<size_t>(b) * p.S + row;
  __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.o) + (tok * p.H + h) * D + CPL * lane;
  if constexpr (CPL == 2) *reinterpret_cast<uint32_t*>(dst) = pk[0];
  else if constexpr (CPL == 4) *reinterpret_cast<uint2*>(dst) = make_uint2(pk[0], pk[1]);
  else *reinterpret_cast<uint4*>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  if (lane == 0 && p.lse != nullptr) p.lse[static_cast<size_t>(hb) * p.S + row] = L * LN2;
}

// Shared memory a VARLEN launch adds: offsets [n_seq + 1], two per-level arrays
// [n_levels + 1], the item count, and the sorted sequence order (16-bit) [n_seq].
constexpr int VARLEN_SMEM_BYTES = ((VARLEN_MAX_SEQ + 1) + 2 * (VARLEN_MAX_LEVELS + 1) + 4) * 4 + VARLEN_MAX_SEQ * 2;

// SPLIT: the launch has a key-split tail (fixed length, not causal).  The other launches use
// the SPLIT = false instantiation, which has none of its code.
template <int D, bool FP8, bool CAUSAL, bool VARLEN, bool SPLIT>
__global__ void __launch_bounds__(AttnCfg<D, FP8>::THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const AttnParams p, const SplitParams sp) {
  using C = AttnCfg<D, FP8>;
  constexpr int NT = C::NT;
  constexpr int NSLOT = C::NSLOT;
  constexpr bool SPLIT_P = NT == 1;    // hand P to the MMA warp in two halves (one query tile)

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  // Fixed-length launches stage O in shared memory for tensor stores; packed batches store rows
  // from registers (a tensor store of a partial tile would write the next sequence's rows).
  constexpr bool STAGE_O = !VARLEN;
  const uint32_t sQ = base_u32;                                  // QBUF x NT tiles
  const uint32_t sKV = base_u32 + C::QBUF * NT * C::TILE_BYTES;  // NSLOT tiles
  const uint32_t sP = sKV + NSLOT * C::TILE_BYTES;               // P_SMEM: NT numerator tiles
  const uint32_t sOst = sP + C::P_BYTES;                         // STAGE_O: O staging
  const uint32_t bar0 = sOst + (STAGE_O ? C::OST_BYTES : 0);     // barriers (8 B each)
  uint8_t* bar_ptr = base + (bar0 - base_u32);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_ptr + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // VARLEN only: offsets; per level, #sequences longer than it (cnt) and its first item (off)
  int* s_cu = reinterpret_cast<int*>(bar_ptr + C::NBAR * 8 + 16);
  int* s_cnt = s_cu + VARLEN_MAX_SEQ + 1;
  int* s_off = s_cnt + VARLEN_MAX_LEVELS + 1;
  int* s_nitems = s_off + VARLEN_MAX_LEVELS + 1;
  int16_t* s_perm = reinterpret_cast<int16_t*>(s_nitems + 4);

  // Q buffer qb: the first pair of barriers, or the pair after everything else
  auto BAR_Q_FULL = [&](int qb) { return qb == 0 ? bar0 : bar0 + 8u * (2 + 2 * NSLOT + 5 * NT + 1); };
  auto BAR_Q_EMPTY = [&](int qb) { return qb == 0 ? bar0 + 8u : bar0 + 8u * (2 + 2 * NSLOT + 5 * NT + 2); };
  auto BAR_KV_FULL = [&](int s) { return bar0 + 8u * (2 + s); };
  auto BAR_KV_EMPTY = [&](int s) { return bar0 + 8u * (2 + NSLOT + s); };
  auto BAR_S_FULL = [&](int t) { return bar0 + 8u * (2 + 2 * NSLOT + t); };
  auto BAR_P_FULL = [&](int t) { return bar0 + 8u * (2 + 2 * NSLOT + NT + t); };
  auto BAR_O_FULL = [&](int t) { return bar0 + 8u * (2 + 2 * NSLOT + 2 * NT + t); };
  auto BAR_O_EMPTY = [&](int t) { return bar0 + 8u * (2 + 2 * NSLOT + 3 * NT + t); };
  auto BAR_MMA_DONE = [&]() { return bar0 + 8u * (2 + 2 * NSLOT + 4 * NT); };
  // the first half of P_t (keys 0..63 of the tile) is in Tensor Memory
  auto BAR_P_HALF = [&](int t) { return bar0 + 8u * (2 + 2 * NSLOT + 4 * NT + 1 + t); };
  // P_SMEM: numerators of tile t in buffer b are in shared memory (4 arrivals).  One barrier
  // per buffer: the softmax warps may run a whole tile ahead of the issuer, and a single
  // barrier could then complete two phases before the issuer looks at it.  A buffer is
  // refilled only after PV_t has read it, so its barrier is never more than one phase ahead.
  auto BAR_P_SM = [&](int t, int b) { return b == 0 ? BAR_P_FULL(t) : BAR_P_HALF(t); };
  // P_SMEM: the softmax warps of tile t have read S_t (4 arrivals), and PV_t has completed
  auto BAR_S_READ = [&](int t) { return bar0 + 8u * (2 + 2 * NSLOT + 5 * NT + 3 + t); };
  auto BAR_PV_DONE = [&](int t) { return bar0 + 8u * (2 + 2 * NSLOT + 6 * NT + 3 + t); };

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();

  if (threadIdx.x == 0) {
    for (int qb = 0; qb < 2; ++qb) {
      mbar_init(BAR_Q_FULL(qb), 1);
      mbar_init(BAR_Q_EMPTY(qb), C::ISSUERS);      // one release per issuer
    }
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(BAR_KV_FULL(s), 1);
      mbar_init(BAR_KV_EMPTY(s), C::ISSUERS);
    }
    for (int t = 0; t < NT; ++t) {
      mbar_init(BAR_S_FULL(t), 1);
      mbar_init(BAR_P_FULL(t), 4);
      mbar_init(BAR_P_HALF(t), 4);
      mbar_init(BAR_O_FULL(t), 1);
      mbar_init(BAR_O_EMPTY(t), 4);
      mbar_init(BAR_S_READ(t), 4);
      mbar_init(BAR_PV_DONE(t), 1);
    }
    mbar_init(BAR_MMA_DONE(), C::ISSUERS);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if constexpr (VARLEN) {
    // Offsets and the length histogram (key = query blocks of a sequence) to shared memory.
    // Offsets that are not 0 .. total, non-decreasing, with every length <= max_seqlen end
    // the launch with ATTN_ERR_INVALID_ARG in the error word before any work is issued.
    constexpr int QR = 128 * NT;                 // query rows per work item
    const int ns = p.n_seq, L = p.n_levels;
    const int tid = static_cast<int>(threadIdx.x);
    int* s_hist = s_off;                         // the histogram, later the per-key counters
    for (int i = tid; i <= ns; i += C::THREADS) s_cu[i] = p.cu_seqlens[i];
    for (int i = tid; i <= L; i += C::THREADS) s_hist[i] = 0;
    __syncthreads();
    bool bad = false;
    for (int sq = tid; sq < ns; sq += C::THREADS) {
      const int len = s_cu[sq + 1] - s_cu[sq];
      if (len < 0 || len > p.max_seqlen) bad = true;
      else if (len > 0) atomicAdd(&s_hist[(len + QR - 1) / QR], 1);
    }
    if (tid == 0) bad |= s_cu[0] != 0 || s_cu[ns] != p.S;
    if (__syncthreads_or(bad)) {
      if (tid == 0 && atomicCAS(p.err_word, 0, 1 /* ATTN_ERR_INVALID_ARG */) == 0) atomicExch(p.err_info, 5);
      return;
    }
    const uint32_t lt_mask = (1u << lane) - 1u;
    if (warp == 0) {
      // cnt[l] = #sequences with more than l query blocks: suffix sums of the histogram,
      // 32 keys at a time from the top
      int carry = 0;
      for (int top = L; top >= 1; top -= 32) {
        const int key = top - static_cast<int>(lane);
        int x = key >= 1 ? s_hist[key] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, x, o);
          if (static_cast<int>(lane) >= o) x += y;
        }
        if (key >= 1) s_cnt[key - 1] = carry + x;
        carry += __shfl_sync(0xffffffffu, x, 31);
      }
      if (lane == 0) s_cnt[L] = 0;
      __syncwarp();
      for (int i = static_cast<int>(lane); i <= L; i += 32) s_hist[i] = 0;
      __syncwarp();
      // stable counting sort by key, descending: position = cnt[key] + earlier equal keys
      for (int base_s = 0; base_s < ns; base_s += 32) {
        const int sq = base_s + static_cast<int>(lane);
        const int len = sq < ns ? s_cu[sq + 1] - s_cu[sq] : 0;
        const int key = (len + QR - 1) / QR;
        const bool act = key > 0;
        const uint32_t grp = __match_any_sync(0xffffffffu, act ? key : -1 - static_cast<int>(lane));
        const int rank = __popc(grp & lt_mask);
        int pos = 0;
        if (act) pos = s_cnt[key] + s_hist[key] + rank;
        __syncwarp();
        if (act) {
          s_perm[pos] = static_cast<int16_t>(sq);
          if (rank == 0) s_hist[key] += __popc(grp);
        }
        __syncwarp();
      }
      // Item offsets, exclusive suffix sums from the top, and the item count.
      //   causal: off[l] = H * #items of the levels above l, an item per (sequence, head) at a
      //           level: x(l) = cnt[l];
      //   else:   off[k] = H * #items of the sequences with more than k blocks, k blocks per
      //           (sequence, head): x(k) = k * (cnt[k-1] - cnt[k]), k >= 1.
      carry = 0;
      const int lmin = CAUSAL ? 0 : 1, lmax = CAUSAL ? L - 1 : L;
      for (int top = lmax; top >= lmin; top -= 32) {
        const int l = top - static_cast<int>(lane);
        const int own = l < lmin ? 0 : (CAUSAL ? s_cnt[l] : l * (s_cnt[l - 1] - s_cnt[l]));
        int x = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, x, o);
          if (static_cast<int>(lane) >= o) x += y;
        }
        if (l >= lmin) s_off[l] = (carry + x - own) * p.H;
        carry += __shfl_sync(0xffffffffu, x, 31);
      }
      if (lane == 0) *s_nitems = carry * p.H;
    }
    __syncthreads();
  }
  if (warp == C::MMA_WARP) tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
  if (warp == C::LOAD_WARP && lane == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    if (STAGE_O) prefetch_tmap(&tmO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---- persistent schedule over work items (query block, head, batch) ----
  // Item order: causal -> heaviest query blocks first; otherwise the query blocks of one head
  // are adjacent (a head's K/V is read from HBM once, then from L2).  CTA k takes item
  // n*G + k in even rounds n and n*G + G-1-k in odd rounds (zig-zag), G = gridDim.x.
  const int HB = p.H * p.B;
  int n_items;
  if constexpr (VARLEN) n_items = *s_nitems;
  else if constexpr (SPLIT) n_items = sp.n_whole + sp.n_tail * sp.n_parts;
  else n_items = p.nQB * HB;
  const int G = static_cast<int>(gridDim.x);
  const int k_cta = static_cast<int>(blockIdx.x);
  auto item_of = [&](int n) { return n * G + ((n & 1) ? (G - 1 - k_cta) : k_cta); };
  // An item: query rows q0 .. q0 + 128 NT - 1 of sequence (b, h), positions counted from the
  // sequence's first token.  VARLEN: the sequence is tokens s0 .. s0 + len - 1 of the packed
  // axis; otherwise it is batch b and len = S (read from the parameters, not kept).
  // sb (VARLEN with FP8): the sequence's first scale block, cu[s] / 128 + s.  SPLIT only: key
  // tiles kt0 .. kt1-1 are the item's (all of them unless it is part `part` of tail block `slot`).
  struct Item { int h, b, q0, hb, nmax, s0, len, sb, kt0, kt1, part, slot; int n[NT]; };
  auto seq_len = [&](const Item& it) {
    if constexpr (VARLEN) return it.len; else return p.S;
  };
  auto key_tiles = [&](const Item& it) {
    if constexpr (VARLEN) return (it.len + 127) / 128; else return p.nK;
  };
  auto tma_row = [&](const Item& it, int r) {    // token coordinate of a tile row in the TMA view
    if constexpr (VARLEN) return it.s0 + r; else return r;
  };
  auto decode = [&](int item, Item& it) {
    int qb;
    if constexpr (SPLIT) {
      it.part = -1;
      it.slot = 0;
    }
    if constexpr (VARLEN) {
      // lowest level (causal) or block count (otherwise) whose first item is <= item
      int lo = CAUSAL ? 0 : 1, hi = CAUSAL ? p.n_levels - 1 : p.n_levels;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s_off[mid] <= item) hi = mid; else lo = mid + 1;
      }
      const int local = item - s_off[lo];
      int sq;
      if constexpr (CAUSAL) {
        sq = s_perm[local / p.H];
        it.h = local % p.H;
        qb = lo;
      } else {
        // sequences with lo blocks occupy sorted ranks cnt[lo] .. cnt[lo-1]-1, H * lo items each
        sq = s_perm[s_cnt[lo] + local / (p.H * lo)];
        const int rem = local % (p.H * lo);
        it.h = rem / lo;
        qb = rem % lo;
      }
      const int s0 = s_cu[sq];
      it.len = s_cu[sq + 1] - s0;
      it.b = 0;
      it.hb = it.h;
      it.s0 = s0;
      it.sb = (s0 >> 7) + sq;
    } else {
      int id = item;
      if constexpr (SPLIT) {
        if (item >= sp.n_whole) {
          const int u = item - sp.n_whole;
          it.part = u / sp.n_tail;
          it.slot = u % sp.n_tail;
          id = sp.n_whole + it.slot;
        }
      }
      if (CAUSAL) {
        qb = p.nQB - 1 - id / HB;
        it.hb = id % HB;
      } else {
        qb = id % p.nQB;
        it.hb = id / p.nQB;
      }
      it.h = it.hb % p.H;
      it.b = it.hb / p.H;
    }
    it.q0 = qb * 128 * NT;
    if constexpr (SPLIT) {
      it.kt0 = 0;
      it.kt1 = key_tiles(it);
      if (it.part >= 0) {
        it.kt0 = it.part * p.nK / sp.n_parts;
        it.kt1 = (it.part + 1) * p.nK / sp.n_parts;
      }
    }
    it.nmax = 0;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int r0 = it.q0 + 128 * t;
      it.n[t] = (r0 >= seq_len(it)) ? 0 : (CAUSAL ? (r0 / 128 + 1) : (SPLIT ? it.kt1 - it.kt0 : key_tiles(it)));
      it.nmax = it.n[t] > it.nmax ? it.n[t] : it.nmax;
    }
  };

  const WaitCtl ctl{p.spin_limit, abort_flag, p.err_word, p.err_info};

  if (warp == C::LOAD_WARP) {
    // ======================================================== TMA producer ==
    if (lane == 0) {
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      int issued = 0, q_issued = 0;
      for (int n = 0; n * G < n_items && !*abort_flag; ++n) {
        const int item = item_of(n);
        if (item >= n_items) break;
        Item it;
        decode(item, it);
        const int kvh = it.h / p.kv_group;     // grouped-query attention: the shared K/V head
        // Q buffer qb is released by the MMA warp after the last S MMA of the item that used it
        // (QBUF items ago).
        const int qb = q_issued % C::QBUF;
        if (!wait_bounded(BAR_Q_EMPTY(qb), ((q_issued / C::QBUF) & 1) ^ 1u, ctl, WHERE_LOAD)) break;
        uint32_t qbytes = 0;
#pragma unroll
        for (int t = 0; t < NT; ++t) qbytes += it.n[t] > 0 ? C::TILE_BYTES : 0;
        mbar_arrive_expect_tx(BAR_Q_FULL(qb), qbytes);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (it.n[t] == 0) continue;
#pragma unroll
          for (int pn = 0; pn < C::NPANEL; ++pn)
            tma_load_4d(sQ + (qb * NT + t) * C::TILE_BYTES + pn * C::PANEL_BYTES, &tmQ, BAR_Q_FULL(qb),
                        pn * C::PANEL_ELEMS, it.h, tma_row(it, it.q0 + 128 * t), it.b, pol_q);
        }
        ++q_issued;
        for (int j = 0; j < it.nmax && !*abort_flag; ++j) {
          for (int kind = 0; kind < 2; ++kind) {
            const int slot = issued % NSLOT;
            const uint32_t phase = (issued / NSLOT) & 1;
            if (!wait_bounded(BAR_KV_EMPTY(slot), phase ^ 1u, ctl, WHERE_LOAD)) break;
            mbar_arrive_expect_tx(BAR_KV_FULL(slot), C::TILE_BYTES);
            const CUtensorMap* m = kind == 0 ? &tmK : &tmV;
#pragma unroll
            for (int pn = 0; pn < C::NPANEL; ++pn)
              tma_load_4d(sKV + slot * C::TILE_BYTES + pn * C::PANEL_BYTES, m, BAR_KV_FULL(slot),
                          pn * C::PANEL_ELEMS, kvh, tma_row(it, 128 * ((SPLIT ? it.kt0 : 0) + j)), it.b, pol_kv);
            ++issued;
          }
        }
      }
      if (*abort_flag) {
        // Drain: every copy still in flight must land before the CTA may exit.
        for (int i = q_issued > C::QBUF ? q_issued - C::QBUF : 0; i < q_issued; ++i)
          wait_drain(BAR_Q_FULL(i % C::QBUF), (i / C::QBUF) & 1, p.spin_limit);
        const int first = issued > NSLOT ? issued - NSLOT : 0;
        for (int i = first; i < issued; ++i)
          wait_drain(BAR_KV_FULL(i % NSLOT), (i / NSLOT) & 1, p.spin_limit);
      }
    }
  } else if (warp >= C::MMA_WARP && warp < C::MMA_WARP + C::ISSUERS) {
    // ========================================================== MMA issuer ==
    if (lane == 0) {
      // Descriptors are built once; a K-step advances the start address field (bits 0-13,
      // in 16-byte units) by adding to the low word.
      const uint64_t dq0 = smem_desc(sQ, 16, C::SBO, C::LAYOUT);
      const uint64_t dkv0 = smem_desc(sKV, 16, C::SBO, C::LAYOUT);
      const uint64_t dv0 = smem_desc(sKV, C::PANEL_BYTES, C::SBO, C::LAYOUT);
      const uint64_t dp0 = smem_desc(sP, 16, 1024, 2);            // P_SMEM: 128-byte rows
      int qsel = 0;              // the Q buffer of the current item
      auto gemm_qk = [&](int t, int slot) {
        const uint32_t d = tmem + 128u * t;
        const uint64_t a0 = dq0 + (((qsel * NT + t) * C::TILE_BYTES) >> 4);
        const uint64_t b0 = dkv0 + ((slot * C::TILE_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS_QK; ++kk) {
          const uint32_t off =
              ((kk / C::STEPS_PER_PANEL) * C::PANEL_BYTES + (kk % C::STEPS_PER_PANEL) * 32) >> 4;
          if (FP8) mma_f8_ss(d, a0 + off, b0 + off, C::IDESC_QK, kk > 0);
          else     mma_f16_ss(d, a0 + off, b0 + off, C::IDESC_QK, kk > 0);
        }
      };
      // O_t += P_t V over K-steps [k_begin, k_end) (each half of the keys follows its own arrival)
      auto gemm_pv = [&](int t, int slot, bool acc, int k_begin, int k_end) {
        const uint32_t d = tmem + 128u * NT + static_cast<uint32_t>(D) * t;
        const uint64_t b0 = dv0 + ((slot * C::TILE_BYTES) >> 4);
#pragma unroll
        for (int kk = k_begin; kk < k_end; ++kk) {
          const uint32_t a = tmem + 128u * t + 8u * kk;
          const uint32_t off = (kk * C::UMMA_K * C::PANEL_ROW) >> 4;
          if (FP8) mma_f8_ts(d, a, b0 + off, C::IDESC_PV, (acc || kk > 0) ? 1u : 0u);
          else     mma_f16_ts(d, a, b0 + off, C::IDESC_PV, (acc || kk > 0) ? 1u : 0u);
        }
      };
      // P_SMEM: O_t += P_t V with P_t from its shared-memory buffer pb, 32 keys per K-step
      auto gemm_pv_smem = [&](int t, int pb, int slot, bool acc) {
        const uint32_t d = tmem + 128u * NT + static_cast<uint32_t>(D) * t;
        const uint64_t a0 = dp0 + (((2 * t + pb) * 128 * 128) >> 4);
        const uint64_t b0 = dv0 + ((slot * C::TILE_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS_PV; ++kk)
          mma_f8_ss(d, a0 + 2 * kk, b0 + ((kk * C::UMMA_K * C::PANEL_ROW) >> 4), C::IDESC_PV,
                    (acc || kk > 0) ? 1u : 0u);
      };
      if constexpr (!C::P_SMEM) {
        // A single issuer: per key step PV_0, S_0, PV_1, S_1 (P_t lies over S_t in Tensor Memory,
        // so S_t(j) follows PV_t(j-1)); with one query tile P is handed over in two halves.
        int consumed = 0;          // K/V ring position
        int pc[NT], ouse[NT];      // P phases consumed, and O uses completed, per query tile
#pragma unroll
        for (int t = 0; t < NT; ++t) pc[t] = ouse[t] = 0;
        bool ok = true;
        for (int n = 0; ok && n * G < n_items; ++n) {
          const int item = item_of(n);
          if (item >= n_items) break;
          Item it;
          decode(item, it);
          qsel = n % C::QBUF;
          ok = wait_bounded(BAR_Q_FULL(qsel), (n / C::QBUF) & 1, ctl, WHERE_MMA);
          if (!ok) break;
          {
            const int ks = consumed % NSLOT;
            ok = wait_bounded(BAR_KV_FULL(ks), (consumed / NSLOT) & 1, ctl, WHERE_MMA);
            ++consumed;
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              if (it.n[t] > 0) {
                gemm_qk(t, ks);
                mma_commit(BAR_S_FULL(t));
              }
            }
            if (it.nmax == 1) mma_commit(BAR_Q_EMPTY(qsel));
            mma_commit(BAR_KV_EMPTY(ks));
          }
          for (int j = 1; ok && j <= it.nmax; ++j) {
            const int vs = consumed % NSLOT;
            ok = wait_bounded(BAR_KV_FULL(vs), (consumed / NSLOT) & 1, ctl, WHERE_MMA);
            ++consumed;
            if (!ok) break;
            tc_fence_after();
            int ks = -1;   // K_j is waited for only right before the first S(j) that needs it
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              if (j - 1 < it.n[t]) {
                if (j - 1 == 0) {
                  // O_t is free once the softmax warps have read the previous item's O_t.
                  if (!wait_bounded(BAR_O_EMPTY(t), (ouse[t] & 1) ^ 1, ctl, WHERE_MMA)) { ok = false; break; }
                }
                if constexpr (SPLIT_P) {
                  if (!wait_bounded(BAR_P_HALF(t), pc[t] & 1, ctl, WHERE_MMA)) { ok = false; break; }
                  tc_fence_after();
                  gemm_pv(t, vs, j - 1 > 0, 0, C::KSTEPS_PV / 2);
                }
                if (!wait_bounded(BAR_P_FULL(t), pc[t] & 1, ctl, WHERE_MMA)) { ok = false; break; }
                ++pc[t];
                tc_fence_after();
                gemm_pv(t, vs, SPLIT_P || j - 1 > 0, SPLIT_P ? C::KSTEPS_PV / 2 : 0, C::KSTEPS_PV);
                if (j - 1 == it.n[t] - 1) {
                  mma_commit(BAR_O_FULL(t));
                  ++ouse[t];
                }
              }
              if (t == NT - 1) mma_commit(BAR_KV_EMPTY(vs));
              if (j < it.n[t]) {
                if (ks < 0) {
                  ks = consumed % NSLOT;
                  if (!wait_bounded(BAR_KV_FULL(ks), (consumed / NSLOT) & 1, ctl, WHERE_MMA)) { ok = false; break; }
                  ++consumed;
                  tc_fence_after();
                }
                gemm_qk(t, ks);
                mma_commit(BAR_S_FULL(t));
              }
            }
            if (ok && ks >= 0) {
              if (j == it.nmax - 1) mma_commit(BAR_Q_EMPTY(qsel));
              mma_commit(BAR_KV_EMPTY(ks));
            }
          }
        }
      } else {
        // P in shared memory: query tile t's issuer.  Every ring position (K_j, V_j of each item, in load order) is
        // released once by each issuer: by a commit after its MMAs that read it, or, where its
        // tile does not need it (causal items, rows past the sequence), by an arrival once the
        // copy has landed, so that the slot's phases stay in step.
        const int t = static_cast<int>(warp) - C::MMA_WARP;
        int consumed = 0;          // K/V ring position
        int pc = 0, ouse = 0;      // P phases consumed, O uses completed
        int qkc = 0;               // QK^T products issued
        bool ok = true;
        auto release = [&](int pos, bool used) -> bool {
          if (used) {
            mma_commit(BAR_KV_EMPTY(pos % NSLOT));
            return true;
          }
          if (!wait_bounded(BAR_KV_FULL(pos % NSLOT), (pos / NSLOT) & 1, ctl, WHERE_MMA)) return false;
          mbar_arrive(BAR_KV_EMPTY(pos % NSLOT));
          return true;
        };
        for (int n = 0; ok && n * G < n_items; ++n) {
          const int item = item_of(n);
          if (item >= n_items) break;
          Item it;
          decode(item, it);
          const int nt = it.n[t];
          qsel = n % C::QBUF;
          if (!wait_bounded(BAR_Q_FULL(qsel), (n / C::QBUF) & 1, ctl, WHERE_MMA)) { ok = false; break; }
          if (nt == 0) mbar_arrive(BAR_Q_EMPTY(qsel));
          // S_t(j) = Q_t K_j^T from ring position kpos; the last one releases the Q buffer.
          auto issue_qk = [&](int j, int kpos) -> bool {
            if (!wait_bounded(BAR_KV_FULL(kpos % NSLOT), (kpos / NSLOT) & 1, ctl, WHERE_MMA)) return false;
            // S_t is free once the softmax warps have read the previous one
            if (qkc > 0 && !wait_bounded(BAR_S_READ(t), (qkc - 1) & 1, ctl, WHERE_MMA)) return false;
            tc_fence_after();
            gemm_qk(t, kpos % NSLOT);
            mma_commit(BAR_S_FULL(t));
            ++qkc;
            if (j == nt - 1) mma_commit(BAR_Q_EMPTY(qsel));
            return true;
          };
          // O_t += P_t(j) V_j from ring position vpos.
          auto issue_pv = [&](int j, int vpos) -> bool {
            if (!wait_bounded(BAR_KV_FULL(vpos % NSLOT), (vpos / NSLOT) & 1, ctl, WHERE_MMA)) return false;
            // O_t is free once the softmax warps have read the previous item's O_t.
            if (j == 0 && !wait_bounded(BAR_O_EMPTY(t), (ouse & 1) ^ 1, ctl, WHERE_MMA)) return false;
            if (!wait_bounded(BAR_P_SM(t, pc & 1), (pc >> 1) & 1, ctl, WHERE_MMA)) return false;
            tc_fence_after();
            gemm_pv_smem(t, pc & 1, vpos % NSLOT, j > 0);
            ++pc;
            mma_commit(BAR_PV_DONE(t));
            if (j == nt - 1) {
              mma_commit(BAR_O_FULL(t));
              ++ouse;
            }
            return true;
          };
          {
            const int kpos = consumed++;
            if (nt > 0 && !issue_qk(0, kpos)) { ok = false; break; }
            if (!release(kpos, nt > 0)) { ok = false; break; }
          }
          for (int j = 1; ok && j <= it.nmax; ++j) {
            const int vpos = consumed++;
            const int kpos = j < it.nmax ? consumed++ : -1;
            const bool do_qk = j < nt, do_pv = j - 1 < nt;
            // S_t(j) first: it needs only the softmax warps to have read S_t(j-1)
            if (do_qk && !issue_qk(j, kpos)) { ok = false; break; }
            if (do_pv && !issue_pv(j - 1, vpos)) { ok = false; break; }
            if (!release(vpos, do_pv)) { ok = false; break; }
            if (kpos >= 0 && !release(kpos, do_qk)) { ok = false; break; }
          }
        }
      }
      // Drain: all issued MMAs complete before Tensor Memory is freed.
      mma_commit(BAR_MMA_DONE());
      wait_drain(BAR_MMA_DONE(), 0, p.spin_limit);
    }
  } else {
    // ============================================================= softmax ==
    const int t = static_cast<int>(warp) / 4;
    const int wq = static_cast<int>(warp) % 4;
    const int row_local = wq * 32 + static_cast<int>(lane);
    const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t s_addr = tl + 128u * t;
    const uint32_t o_addr = tl + 128u * NT + static_cast<uint32_t>(D) * t;
    int sc = 0, ouse = 0;      // S phases consumed, O uses completed (this tile)
    int pcnt = 0;              // P_SMEM: numerator tiles handed over (this tile)
    // P_SMEM: this thread's row of P_t in buffer 0, 128 bytes in the 128-byte swizzle (16-byte
    // chunk c of row r at chunk c ^ (r & 7) of its row); P_t number k goes to buffer k & 1
    const uint32_t p_row = sP + static_cast<uint32_t>(2 * t) * (128u * 128u) +
                           static_cast<uint32_t>((row_local >> 3) * 1024 + (row_local & 7) * 128);
    bool ok = true;
    for (int n = 0; ok && n * G < n_items; ++n) {
      const int item = item_of(n);
      if (item >= n_items) break;
      Item it;
      decode(item, it);
      const int r0 = it.q0 + 128 * t;
      const int nt = SPLIT ? it.n[t] : ((r0 >= seq_len(it)) ? 0 : (CAUSAL ? (r0 / 128 + 1) : key_tiles(it)));
      if (nt == 0) continue;
      const int row = it.q0 + 128 * t + row_local;
      // FP8 block scales: (b*H + h) * nK; the K/V ones belong to the shared key/value head,
      // (b * Hkv + h / G) * nK.  VARLEN: h * stride + the sequence's first block.
      const size_t blk_base = VARLEN ? static_cast<size_t>(it.h) * p.scale_stride + it.sb
                                     : static_cast<size_t>(it.hb) * p.nK;
      const size_t kv_base = VARLEN ? blk_base
                                    : static_cast<size_t>(it.b * (p.H / p.kv_group) + it.h / p.kv_group) * p.nK;

      float sq = 1.f, sv_max = 1.f;
      if (FP8) {
        if (p.q_scale != nullptr) sq = p.q_scale[blk_base + (it.q0 + 128 * t) / 128];
        if (p.v_scale != nullptr) {
          sv_max = 0.f;
          const int j0 = SPLIT ? it.kt0 : 0, j1 = SPLIT ? it.kt1 : key_tiles(it);
          for (int j = j0 + static_cast<int>(lane); j < j1; j += 32) sv_max = fmaxf(sv_max, p.v_scale[kv_base + j]);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) sv_max = fmaxf(sv_max, __shfl_xor_sync(0xffffffffu, sv_max, o));
          sv_max = fmaxf(sv_max, 0x1p-96f);  // every value scale 0: O = 0, l still counts
        }
      }

      // SPLIT: this item's key tiles start at kt0; without the causal mask only the sequence's
      // last key tile can be ragged, and it is the item's last tile when the item reaches it
      const size_t kv_tile0 = kv_base + (SPLIT ? it.kt0 : 0);
      const bool ragged_end = SPLIT && it.kt1 == key_tiles(it) && (seq_len(it) & 127) != 0;

      float m_run = -INFINITY;
      float l_run = 0.f;
      // FP8 per-key-tile factors, lane l holding those of tile 32 (j / 32) + l: the exponent
      // multiplier c_log2 sq sk, the numerators' offset bias = log2(sv / sv_max) (V's block scale
      // relative to the largest, folded into P) and 2^-bias, which takes it out of the row sum.
      // A zero scale (a block of zeros) counts as 2^-30 of the largest: its numerators vanish in
      // E4M3, the row sum still takes them at full weight.  The raw scales of the next 32 tiles
      // are read 32 tiles ahead, so their latency hides behind the loop.
      float cm_l = 1.f, bias_l = 0.f, ir_l = 1.f, skr_next = 1.f, svr_next = 1.f;
      const float csq = p.c_log2 * sq, sv_floor = sv_max * 0x1p-30f, lg_svmax = __log2f(sv_max);
      auto read_raw = [&](int jb, float& skr, float& svr) {
        const int jj = jb + static_cast<int>(lane);
        skr = 1.f;
        svr = 1.f;
        if (jj < nt) {
          if (p.k_scale != nullptr) skr = p.k_scale[kv_tile0 + jj];
          if (p.v_scale != nullptr) svr = p.v_scale[kv_tile0 + jj];
        }
      };
      auto derive = [&](float skr, float svr) {
        cm_l = csq * skr;
        bias_l = __log2f(fmaxf(svr, sv_floor)) - lg_svmax;
        ir_l = ex2(-bias_l);
      };
      float cm_n = p.c_log2, bias_n = 0.f, ir_n = 1.f;    // FP8: tile j's factors, fetched a tile ahead
      if (FP8) {
        float skr, svr;
        read_raw(0, skr, svr);
        derive(skr, svr);
        if (nt > 32) read_raw(32, skr_next, svr_next);
        cm_n = __shfl_sync(0xffffffffu, cm_l, 0);
        bias_n = __shfl_sync(0xffffffffu, bias_l, 0);
        ir_n = __shfl_sync(0xffffffffu, ir_l, 0);
      }
      for (int j = 0; j < nt; ++j) {
        float cmul = p.c_log2, bias = 0.f, inv_r = 1.f;
        if (FP8) {
          cmul = cm_n;
          bias = bias_n;
          inv_r = ir_n;
          const int jn = j + 1;
          if ((jn & 31) == 0 && jn < nt) {
            derive(skr_next, svr_next);
            if (jn + 32 < nt) read_raw(jn + 32, skr_next, svr_next);
          }
          cm_n = __shfl_sync(0xffffffffu, cm_l, jn & 31);
          bias_n = __shfl_sync(0xffffffffu, bias_l, jn & 31);
          ir_n = __shfl_sync(0xffffffffu, ir_l, jn & 31);
        }
        if (!warp_wait(BAR_S_FULL(t), sc & 1, ctl, WHERE_SOFTMAX)) { ok = false; break; }
        ++sc;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + 32u * c, sr[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) reg_fence(sr[c][i]);
        if constexpr (C::P_SMEM) {
          // S_t is in registers: the MMA warp may compute the next S_t over it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR_S_READ(t));
        }

        // masks: causal diagonal tile, or the ragged last key tile
        if (SPLIT ? (j == nt - 1 && ragged_end)
                  : (CAUSAL ? (j == nt - 1) : (j == key_tiles(it) - 1 && (seq_len(it) & 127) != 0))) {
          // last visible column
          const int lim = CAUSAL ? (row - 128 * j) : (SPLIT ? ((seq_len(it) - 1) & 127) : (seq_len(it) - 128 * j - 1));
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (32 * c + i > lim) sr[c][i] = __float_as_uint(-INFINITY);
        }

        float mx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = __uint_as_float(sr[k / 2][(k % 2) * 16]);
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const int k = (c * 2 + i / 16) & 7;
            mx[k] = max3(mx[k], __uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1]));
          }
        const float m_tile =
            max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * cmul;

        bool rescale = false;
        float alpha = 1.f;
        if (j == 0) {
          m_run = m_tile;
        } else if (m_tile > m_run + TAU) {
          alpha = ex2(m_run - m_tile);
          m_run = m_tile;
          l_run *= alpha;
          rescale = true;
        }

        const float nb = bias - m_run;
        const uint64_t c2 = f2_pack(cmul, cmul);
        const uint64_t nb2 = f2_pack(nb, nb);
        uint64_t ls2[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) ls2[k] = f2_pack(0.f, 0.f);
        // O_t holds PV_t(j-1) complete (it preceded S_t(j), or P_SMEM: PV-done) and PV_t(j) waits
        // for this warp's arrival, so O_t is rescaled in place before that arrival.  With one query tile
        // (SPLIT_P) the first 64 keys' numerators are handed over on their own, so PV over them
        // overlaps the exponentials of the second half; with two tiles the other tile's MMAs
        // already fill that time and the extra hand-off only costs.
        auto rescale_o = [&]() -> bool {
          if (__any_sync(0xffffffffu, rescale)) {
            // P_SMEM: S_t(j) does not follow PV_t(j-1), so O_t waits for it here
            if (C::P_SMEM && pcnt > 0 && !warp_wait(BAR_PV_DONE(t), (pcnt - 1) & 1, ctl, WHERE_SOFTMAX))
              return false;
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(o_addr + 32u * c, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                reg_fence(o[i]);
                o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              }
              tmem_st32(o_addr + 32u * c, o);
            }
          }
          return true;
        };
        auto hand_off_first_half = [&]() {
          (void)rescale_o();
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR_P_HALF(t));
        };
        if (!FP8) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1])), c2, nb2);
              float x0, x1;
              f2_unpack(x2, x0, x1);
              const float p0 = ex2(x0), p1 = ex2(x1);
              ls2[i & 3] = f2_add(ls2[i & 3], f2_pack(p0, p1));
              pk[i] = pack_bf16x2(p0, p1);
            }
            tmem_st16(s_addr + 16u * c, pk);
            if (SPLIT_P && c == 1) hand_off_first_half();
          }
        } else {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float pv[4];
#pragma unroll
              for (int e = 0; e < 4; e += 2) {
                const int col = 64 * h2 + 4 * i + e;
                const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(sr[col / 32][col % 32]),
                                                   __uint_as_float(sr[col / 32][col % 32 + 1])), c2, nb2);
                float x0, x1;
                f2_unpack(x2, x0, x1);
                pv[e] = ex2(x0);
                pv[e + 1] = ex2(x1);
                ls2[(2 * i + e / 2) & 3] = f2_add(ls2[(2 * i + e / 2) & 3], f2_pack(pv[e], pv[e + 1]));
              }
              pk[i] = pack_e4m3x4(pv[0], pv[1], pv[2], pv[3]);
            }
            if constexpr (C::P_SMEM) {
              // The buffer's previous numerators (two tiles back) have been read: the MMA warp
              // issued S_t(j), whose completion this warp has seen, after PV_t(j - 2).
              const uint32_t prow = p_row + static_cast<uint32_t>(pcnt & 1) * (128u * 128u);
#pragma unroll
              for (int c4 = 0; c4 < 4; ++c4) {
                const uint32_t chunk = static_cast<uint32_t>((4 * h2 + c4) ^ (row_local & 7));
                st_shared_v4(prow + 16u * chunk, pk[4 * c4], pk[4 * c4 + 1], pk[4 * c4 + 2], pk[4 * c4 + 3]);
              }
            } else {
              tmem_st16(s_addr + 16u * h2, pk);
              if (SPLIT_P && h2 == 0) hand_off_first_half();
            }
          }
        }
        {
          const uint64_t t2 = f2_add(f2_add(ls2[0], ls2[1]), f2_add(ls2[2], ls2[3]));
          float a0, a1;
          f2_unpack(t2, a0, a1);
          l_run += (a0 + a1) * inv_r;
        }
        if (!SPLIT_P && !rescale_o()) { ok = false; break; }
        tmem_wait_st();
        const uint32_t bar_p = C::P_SMEM ? BAR_P_SM(t, pcnt & 1) : BAR_P_FULL(t);
        if constexpr (C::P_SMEM) {
          fence_proxy_async_smem();      // P_t's shared-memory writes, for the tensor core
          ++pcnt;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_p);
      }
      if (!ok) break;

      // ---- epilogue: O / l -> bf16, lse; then hand O_t back to the MMA warp ----
      if (!warp_wait(BAR_O_FULL(t), ouse & 1, ctl, WHERE_SOFTMAX)) { ok = false; break; }
      ++ouse;
      tc_fence_after();
      const float inv_l = sv_max / l_run;
      const bool valid = row < seq_len(it);
      // token of this row on O's token axis (packed axis, or b * S + row)
      size_t tok;
      if constexpr (VARLEN) tok = static_cast<size_t>(it.s0) + (valid ? row : 0);
      else tok = static_cast<size_t>(it.b) * p.S + (valid ? row : 0);
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + (tok * p.H + it.h) * D;
      if constexpr (SPLIT) {
        // a key range of a cut block (recomputed from n: nothing of it stays live in the loop)
        const int u = item_of(n) - sp.n_whole;
        if (u >= 0) {
          const int wrow0 = it.q0 + 128 * t + 32 * wq;   // this warp's first row
          split_store<D, NT>(sp, u % sp.n_tail, u / sp.n_tail, t, row_local, valid, o_addr, inv_l,
                             m_run + __log2f(l_run), BAR_O_EMPTY(t),
                             sOst + static_cast<uint32_t>(warp) * C::OST_WARP_BYTES,
                             seq_len(it) - wrow0);
          continue;
        }
      }
      // this warp's 32 rows of the tile: the first one, and its staging buffers
      const int row0 = it.q0 + 128 * t + 32 * wq;
      const uint32_t ost = sOst + static_cast<uint32_t>(warp) * C::OST_WARP_BYTES;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(o_addr + 32u * c, o);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          reg_fence(o[2 * i]);
          reg_fence(o[2 * i + 1]);
          pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
        }
        if constexpr (STAGE_O) {
          // buffer c & 1 is free once at most one store (chunk c - 1's) still reads its buffer;
          // at chunk 0 the item before's last stores (same buffers) must have read them all
          if (lane == 0) {
            if (c == 0) bulk_wait_read_all();
            else if (c >= 2) bulk_wait_read_1();
          }
          __syncwarp();
          const uint32_t buf = ost + (c & 1) * (32 * 64);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            // row = lane (64 bytes), 16-byte chunk v4, 64-byte swizzle: chunk ^ ((row >> 1) & 3)
            const uint32_t addr = buf + lane * 64 + ((v4 ^ ((lane >> 1) & 3)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * v4]),
                         "r"(pk[4 * v4 + 1]), "r"(pk[4 * v4 + 2]), "r"(pk[4 * v4 + 3])
                         : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
          // rows beyond S are clipped by the store; a warp whose rows all lie beyond S stores none
          if (lane == 0 && row0 < seq_len(it)) {
            tma_store_4d(&tmO, buf, 32 * c, it.h, row0, it.b);
            bulk_commit_group();
          }
        } else if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR_O_EMPTY(t));
      if (valid && p.lse != nullptr)
        p.lse[static_cast<size_t>(it.hb) * p.S + tma_row(it, row)] = (m_run + __log2f(l_run)) * LN2;
    }
  }

  // the epilogue's tensor stores have read their staging buffers (and written O) before the
  // CTA's shared memory goes away
  if (STAGE_O && warp < C::NUM_SOFTMAX_WARPS && lane == 0) bulk_wait_all();
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool FP8, bool CAUSAL, bool VARLEN>
cudaError_t launch_attn(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& to, const AttnParams& p, cudaStream_t stream,
                        const SplitParams* split_plan) {
  using C = AttnCfg<D, FP8>;
  constexpr int SMEM = C::SMEM_BYTES + (VARLEN ? VARLEN_SMEM_BYTES : C::OST_BYTES);
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  constexpr bool CAN_SPLIT = !CAUSAL && !VARLEN;
  const bool split = CAN_SPLIT && split_plan != nullptr && split_plan->n_parts > 1;
  const SplitParams sp = split ? *split_plan : SplitParams{0, 0, 1, nullptr, nullptr};
  static std::atomic<unsigned long long> configured{0};   // one bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if ((configured.load() & bit) == 0) {
    e = cudaFuncSetAttribute(attn_fwd_kernel<D, FP8, CAUSAL, VARLEN, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    if constexpr (CAN_SPLIT) {
      e = cudaFuncSetAttribute(attn_fwd_kernel<D, FP8, CAUSAL, VARLEN, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
      if (e != cudaSuccess) return e;
    }
    configured.fetch_or(bit);
  }
  static int sm_count[64] = {0};
  if (sm_count[dev & 63] == 0) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sm_count[dev & 63] = n;
  }
  // VARLEN: an upper bound (every sequence adds at most one partial query block per head)
  const long long items = VARLEN ? (static_cast<long long>(p.S) / (128 * C::NT) + p.n_seq) * p.H
                         : split ? static_cast<long long>(sp.n_whole) + 1ll * sp.n_tail * sp.n_parts
                                 : static_cast<long long>(p.nQB) * p.H * p.B;
  const long long grid = items < sm_count[dev & 63] ? items : sm_count[dev & 63];   // persistent
  if constexpr (CAN_SPLIT) {
    if (split) {
      attn_fwd_kernel<D, FP8, CAUSAL, VARLEN, true>
          <<<static_cast<unsigned>(grid), C::THREADS, SMEM, stream>>>(tq, tk, tv, to, p, sp);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      const long long warps = static_cast<long long>(sp.n_tail) * 128 * C::NT;
      split_merge_kernel<D, C::NT><<<static_cast<unsigned>((warps + 7) / 8), 256, 0, stream>>>(p, sp);
      return cudaGetLastError();
    }
  }
  attn_fwd_kernel<D, FP8, CAUSAL, VARLEN, false>
      <<<static_cast<unsigned>(grid), C::THREADS, SMEM, stream>>>(tq, tk, tv, to, p, sp);
  return cudaGetLastError();
}

}  // namespace ea46
