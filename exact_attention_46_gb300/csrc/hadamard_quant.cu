// hadamard_quant.cu -- random-sign Hadamard rotation + per-block E4M3 quantisation.
//
// What it computes ("FlashAttention-3 (NL)", "Technische innovaties", item 3; hada.io FA3
// summary, "Niedrige FP8-Präzision und incoherent processing"): every D-element row x of a
// [B, S, H, D] bf16 tensor becomes x' = (x * signs) H_D / sqrt(D) (H_D the Sylvester
// Hadamard matrix; no rotation when signs is null), each (b, h, 128-token block) gets one
// scale = amax(|x'|) / 448 (1 for an all-zero block), and out = E4M3(x' / scale), rounded to
// nearest even and saturating.  The rounded quotient is formed in fp32 as
// y * (448 / amax(y)) with y = (x * signs) H_D the unnormalised transform.
//
// Design: the transform is O(D log D) per row and the kernel is bound by HBM traffic
// (2 bytes read + 1 byte written per element) once its instruction count is low, so it stays
// on the FP32 pipes: no tensor cores.  One persistent CTA per SM streams blocks of 128 rows
// through a ring of NSTAGE shared-memory stages filled by TMA (the same 128-byte-swizzled box
// the attention kernel uses).  The CTA's threads form G groups of one block's worth of threads;
// group g takes every G-th block and synchronises on a named barrier of its own.  A stage is
// refilled with the block NSTAGE further on as soon as its group holds the values in
// registers -- before the transform -- so about NSTAGE loads stay in flight per SM whatever
// the groups are doing.  A thread owns a row (lanes l and l + 16 share one at D = 256), so the
// butterfly stages run in registers (plus one lane-shuffle stage at D = 256); the 8 lanes of
// a 128-bit read phase hold 8 rows and read the same 16-byte chunk of each, which the swizzle
// makes conflict-free.  The random signs are applied as XOR masks on the packed bf16 words,
// read from a small shared-memory table by broadcast.  Rows beyond S arrive zero-filled.  The
// codes go into the group's own output buffer in the swizzled layout of the E4M3 output map
// and leave with one tensor store per panel (rows beyond S clipped), so L2 sees whole lines;
// the buffer is reused once that store has read it.
//
// Rotary embedding fused in front (hada.io FA3 summary, same section: the transform is
// bandwidth-bound and costs nothing extra when fused with a preceding bandwidth-bound op such
// as rotary embedding).  RoPE as in RoFormer (Su et al. 2021, section 3.2): pair
// (x[2i], x[2i+1]) of the row at position p turns by p * theta_i, before the signs and the
// transform, with no rounding in between.  A 128-row block would need 128 table rows (4 D
// bytes each, twice the block's own input), so the kernel rebuilds (cos, sin)(p theta_i) with
// the angle-addition identity, as the complex product of table row 128 blk + 16 r1 (8 rows per
// block, bulk-copied into the block's stage after its input) and table row r0 (16 rows,
// resident), r = 16 r1 + r0.
//
// Packed variable-length batches (VARLEN): x is [total, H, D] with sequence offsets cu_seqlens,
// and a block never straddles two sequences -- sequence s is cut into 128-token blocks from its
// own first token.  Block k of sequence s has scale index cu[s] / 128 + s + k (no two sequences
// share one; at most one index per sequence stays unused), so a work item is (index, head) and
// a binary search over the strictly increasing cu[s] / 128 + s finds its sequence.  Rows past
// the sequence's end arrive with the box but count as zero; a whole block leaves by tensor
// store, a partial one row by row from registers (a tensor store would overwrite the next
// sequence's rows).  The offsets are checked before anything is written.  With RoPE the
// positions restart at every sequence's first token (the table rows of block k of a sequence
// are those of block k of a tensor of its own), and a table too short for some sequence is an
// error found in the same check.
#include <atomic>
#include <cstdint>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ea46 {

namespace {

constexpr int QROWS = 128;            // tokens per scale block
constexpr int NCOARSE = 8;            // rotary rows 128 blk + 16 r1 per block
constexpr int NFINE = 16;             // rotary rows r0 = 0..15, resident

template <int D, bool ROPE, bool ROTATE = true, bool VARLEN = false>
struct QCfg {
  static constexpr int VPT = D < 128 ? D : 128;                            // values per thread
  static constexpr int TPR = D / VPT;                                      // threads per row
  static constexpr int RPW = 32 / TPR;                                     // rows per warp
  static constexpr int GTHREADS = QROWS * TPR;                             // threads of one group
  static constexpr int GWARPS = GTHREADS / 32;
  // groups per CTA (one CTA per SM): as many 128-row blocks in registers at once as the
  // register file holds
  // (three groups of the rotary forms at D = 128 fit 170 registers only for the rotated,
  // fixed-length one; the others keep two)
  static constexpr int G = D == 64 ? 4 : (D == 128 ? (ROPE && (!ROTATE || VARLEN) ? 2 : 3) : 1);
  static constexpr int THREADS = G * GTHREADS;
  static constexpr int ROW_BYTES = D * 2;                                  // bf16 row
  static constexpr int PANEL_BYTES = 128 * 128;                            // 128 rows x 128 B
  static constexpr int NPANEL = ROW_BYTES / 128;                           // 1, 2, 4
  static constexpr int IN_BYTES = QROWS * ROW_BYTES;
  // rotary table rows in shared memory: (cos, sin) pairs, 8 bytes each, a thread's VPT/2 pairs
  // at part * SEG_BYTES; rows padded by 16 bytes so that the 8 rows of one 128-bit read phase
  // fall in distinct banks.  A block's 8 coarse rows travel in its stage, after the input.
  static constexpr int SEG_BYTES = 4 * VPT;
  static constexpr int TROW = 4 * D + 16;
  static constexpr int COARSE_OFF = IN_BYTES;
  static constexpr int STAGE_BYTES = (IN_BYTES + (ROPE ? NCOARSE * TROW : 0) + 1023) / 1024 * 1024;
  static constexpr int NSTAGE = D == 64 ? (ROPE ? 8 : 10) : (D == 128 ? (ROPE ? 4 : 5) : 2);
  // E4M3 codes of a block, staged for one tensor store per 128-byte panel (64-byte rows with a
  // 64-byte swizzle at D = 64), one buffer per group
  static constexpr int CODE_PANEL = D < 128 ? D : 128;                     // bytes per code row
  static constexpr int NCPANEL = D / CODE_PANEL;
  static constexpr int OUT_BYTES = QROWS * D;
  static constexpr int OFF_OUT = NSTAGE * STAGE_BYTES;
  static constexpr int OFF_FINE = OFF_OUT + G * OUT_BYTES;
  // packed-bf16 sign XOR masks [D/2] without RoPE; per-pair masks sign(2i) != sign(2i+1) [D/2]
  // with it (the even element's sign is folded into the resident rotary rows)
  static constexpr int OFF_SIGN = OFF_FINE + (ROPE ? NFINE * TROW : 0);
  static constexpr int SIGN_BYTES = 2 * D;
  static constexpr int OFF_BAR = OFF_SIGN + SIGN_BYTES;
  static constexpr int OFF_WMAX = OFF_BAR + 8 * NSTAGE;                    // [G][2][GWARPS] floats
  static constexpr int OFF_ISSUED = OFF_WMAX + G * 2 * GWARPS * 4;         // [NSTAGE] loads issued
  static constexpr int OFF_GEN = OFF_ISSUED + 4 * NSTAGE;                  // [NSTAGE] block in the stage
  static constexpr int OFF_TAKEN = OFF_GEN + 4 * NSTAGE;                   // [NSTAGE] warps done reading
  static constexpr int OFF_ABORT = OFF_TAKEN + 4 * NSTAGE;
  static constexpr int OFF_INFO = (OFF_ABORT + 16 + 7) / 8 * 8;           // VARLEN: [NSTAGE] (tok0, rows)
  static constexpr int SMEM_BYTES = 1024 + OFF_INFO + 8 * NSTAGE;
  static constexpr uint32_t TX_BYTES = IN_BYTES + (ROPE ? NCOARSE * 4 * D : 0);
  static_assert(TPR >= 1 && TPR <= 2 && D % VPT == 0, "row split");
  static_assert(G <= 4, "named barriers 1 .. G");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(STAGE_BYTES % 1024 == 0 && OFF_OUT % 1024 == 0 && OUT_BYTES % 1024 == 0,
                "swizzled tiles start on 1024-byte boundaries");
  static_assert(OFF_FINE % 16 == 0 && OFF_SIGN % 16 == 0 && OFF_BAR % 8 == 0 && (IN_BYTES + TROW) % 16 == 0,
                "alignment");
};

__device__ __forceinline__ float4 lds128(uint32_t addr) {
  float4 f;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(f.x), "=f"(f.y), "=f"(f.z), "=f"(f.w) : "r"(addr));
  return f;
}

// Pair (v0, v1) turned by the angle whose (cos, sin) is the complex product of (ac, as)
// and (fc, fs).
__device__ __forceinline__ void rotary_pair(float& v0, float& v1, float ac, float as, float fc, float fs) {
  const float c = ac * fc - as * fs;
  const float s = as * fc + ac * fs;
  const float x0 = v0, x1 = v1;
  v0 = x0 * c - x1 * s;
  v1 = x0 * s + x1 * c;
}

__device__ __forceinline__ int ld_acquire_shared(uint32_t addr) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_shared(uint32_t addr, int v) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Count one arrival at a shared counter (acquire + release); returns the count before it.
__device__ __forceinline__ uint32_t atom_add_acq_rel_shared(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}

// Barrier `id` over the n threads of one group, returning whether any of them passed true.
__device__ __forceinline__ bool group_bar_or(uint32_t id, uint32_t n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// QKV: the three tensors Q, K, V in one launch (blocks of tensor t numbered after tensor t-1's),
// the first p.rot_tensors of them rotated: one ramp and one tail instead of three.
template <int D, bool ROTATE, bool ROPE, bool VARLEN, bool QKV>
__global__ void __launch_bounds__(QCfg<D, ROPE, ROTATE, VARLEN>::THREADS, 1)
    hadamard_quant_kernel(const __grid_constant__ QuantMaps m, const QuantParams p) {
  using C = QCfg<D, ROPE, ROTATE, VARLEN>;
  static_assert(!QKV || (ROTATE && !ROPE && !VARLEN), "the three-tensor form is fixed-length, without RoPE");
  constexpr int VPT = C::VPT;
  constexpr int NSTAGE = C::NSTAGE;
  constexpr int NW = VPT / 8;         // 16-byte input chunks per thread

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  uint32_t* sign_mask = reinterpret_cast<uint32_t*>(base + C::OFF_SIGN);
  const uint32_t bar0 = base_u32 + C::OFF_BAR;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + C::OFF_ABORT);
  int* issued = reinterpret_cast<int*>(base + C::OFF_ISSUED);              // loads per stage
  const uint32_t gen0 = base_u32 + C::OFF_GEN;                             // block each stage holds
  uint32_t* taken = reinterpret_cast<uint32_t*>(base + C::OFF_TAKEN);    // warps done with each stage
  int2* stage_info = reinterpret_cast<int2*>(base + C::OFF_INFO);         // VARLEN: (tok0, rows)

  // Groups of GTHREADS threads each take every G-th block of this CTA; a group synchronises on
  // its own named barrier (1 + g), never with the other groups.
  const int g = static_cast<int>(threadIdx.x) / C::GTHREADS;
  const int gt = static_cast<int>(threadIdx.x) % C::GTHREADS;
  const bool leader = gt == 0;
  const uint32_t gbar = 1u + static_cast<uint32_t>(g);
  const int gwarp = gt >> 5, lane = threadIdx.x & 31;
  float* warp_max = reinterpret_cast<float*>(base + C::OFF_WMAX) + g * 2 * C::GWARPS;   // [2][GWARPS]
  const uint32_t outbuf = base_u32 + C::OFF_OUT + g * C::OUT_BYTES;
  // row and the part of it this thread owns: a warp holds RPW rows, lanes l, l + RPW, ... share
  // a row, so the 8 lanes of one 128-bit shared-memory read phase hold 8 different rows
  const int r = gwarp * C::RPW + lane % C::RPW;
  const int part = lane / C::RPW;
  const int nb1 = p.nblk * p.H * p.B;                 // blocks of one tensor
  const int nblocks = nb1 * (QKV ? 3 : 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(bar0 + 8u * s, 1);
      issued[s] = 0;
      taken[s] = 0;
      st_release_shared(gen0 + 4u * s, -1);
    }
    *abort_flag = 0;
    fence_barrier_init();
    for (int t = 0; t < (QKV ? 3 : 1); ++t) {
      prefetch_tmap(&m.x[t]);
      prefetch_tmap(&m.out[t]);
    }
  }

  // Load of the k-th block of this CTA into stage k % NSTAGE.  Called by thread 0 for the first
  // NSTAGE blocks, then by lane 0 of the last warp of the group that has just taken block
  // k - NSTAGE out of that stage: one caller per stage at a time.
  auto issue = [&](int k) {
    const int bt = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
    const int tsr = QKV ? bt / nb1 : 0, bi = bt - tsr * nb1;
    const int h = bi % p.H, blk = (bi / p.H) % p.nblk, b = bi / (p.H * p.nblk);
    const int s = k % NSTAGE;
    const uint32_t st = base_u32 + s * C::STAGE_BYTES;
    const uint32_t bar = bar0 + 8u * s;
    issued[s] += 1;
    int tok0 = blk * QROWS, rblk = blk;   // rblk: the block's position block for RoPE
    // the stage's next phase is block k's; published before the arrival (release), so that a
    // waiter that sees k here sees the barrier at or past the phase block k's load completes
    if constexpr (VARLEN) {
      // the sequence of index blk: the last s with cu[s] / 128 + s <= blk (cu[0] / 128 + 0 = 0)
      int lo = 0, hi = p.n_seq - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((p.cu_seqlens[mid] >> 7) + mid <= blk) lo = mid; else hi = mid - 1;
      }
      const int s0 = p.cu_seqlens[lo], len = p.cu_seqlens[lo + 1] - s0;
      const int kb = blk - ((s0 >> 7) + lo);
      const int rows = 128 * kb < len ? min(QROWS, len - 128 * kb) : 0;
      tok0 = s0 + 128 * kb;
      rblk = kb;
      stage_info[s] = make_int2(tok0, rows);
      if (rows == 0) {                // an index no block lives at
        st_release_shared(gen0 + 4u * s, k);
        mbar_arrive(bar);
        return;
      }
    }
    st_release_shared(gen0 + 4u * s, k);
    mbar_arrive_expect_tx(bar, C::TX_BYTES);
#pragma unroll
    for (int pn = 0; pn < C::NPANEL; ++pn)
      tma_load_4d(st + pn * C::PANEL_BYTES, &m.x[tsr], bar, 64 * pn, h, tok0, b,
                  l2_policy_evict_first());
    if (ROPE) {
      // coarse rows 128 blk + 16 r1 after the block's input in the same stage
#pragma unroll
      for (int r1 = 0; r1 < NCOARSE; ++r1)
        bulk_load(st + C::COARSE_OFF + r1 * C::TROW,
                  p.rope_cs + static_cast<size_t>(rblk * QROWS + 16 * r1) * D, 4 * D, bar,
                  l2_policy_evict_last());
    }
  };
  const int my_blocks = (nblocks - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                        static_cast<int>(gridDim.x);
  // This grid may be launched while the previous grid on the stream is still running
  // (programmatic dependent launch), and that grid may have produced x, the signs, the offsets
  // or the rotary table: nothing is read from global memory before it has completed.  What
  // comes before this point (barrier set-up, tensor-map prefetch) overlaps its tail.
  grid_dependency_wait();
  // Fixed-length launches start their first loads at once, before the tables below (whose
  // global reads would otherwise delay them); packed batches check their offsets first.
  if (!VARLEN && threadIdx.x == 0)
    for (int k = 0; k < NSTAGE && k < my_blocks; ++k) issue(k);
  if (!ROPE) {
    // bit 15 flips the even element of a packed bf16 pair, bit 31 the odd one
    for (int w = static_cast<int>(threadIdx.x); w < D / 2; w += C::THREADS)
      sign_mask[w] = ROTATE && p.signs != nullptr ? ((p.signs[2 * w] < 0.f ? 0x00008000u : 0u) |
                                                     (p.signs[2 * w + 1] < 0.f ? 0x80000000u : 0u))
                                                  : 0u;
  } else {
    // The rotary step comes before the signs: the even element's sign is folded into the
    // resident rows below, the odd element then needs sign(2i) * sign(2i+1).
    for (int w = static_cast<int>(threadIdx.x); w < D / 2; w += C::THREADS)
      sign_mask[w] = ROTATE && ((p.signs[2 * w] < 0.f) != (p.signs[2 * w + 1] < 0.f)) ? 0x80000000u : 0u;
    // resident rotary rows 0..15, times the even element's sign
    for (int idx = static_cast<int>(threadIdx.x); idx < NFINE * (D / 2); idx += C::THREADS) {
      const int f = idx / (D / 2), i = idx % (D / 2);
      float2 cs = reinterpret_cast<const float2*>(p.rope_cs)[idx];
      if (ROTATE && p.signs[2 * i] < 0.f) cs = make_float2(-cs.x, -cs.y);
      *reinterpret_cast<float2*>(base + C::OFF_FINE + f * C::TROW + 8 * i) = cs;
    }
  }
  if constexpr (VARLEN) {
    // offsets that are not 0 .. total, non-decreasing: nothing is written
    bool bad = false;
    for (int i = static_cast<int>(threadIdx.x); i < p.n_seq; i += C::THREADS) {
      const int len = p.cu_seqlens[i + 1] - p.cu_seqlens[i];
      bad |= len < 0;
      if (ROPE) bad |= static_cast<long long>(len + QROWS - 1) / QROWS * QROWS > p.n_pos;
    }
    if (threadIdx.x == 0) bad |= p.cu_seqlens[0] != 0 || p.cu_seqlens[p.n_seq] != p.S;
    if (__syncthreads_or(bad)) {
      grid_launch_dependents();
      if (threadIdx.x == 0 && atomicCAS(p.err_word, 0, 1 /* ATTN_ERR_INVALID_ARG */) == 0) atomicExch(p.err_info, 11);
      return;
    }
  }
  __syncthreads();
  // The next grid on the stream may start its own set-up on the SMs this grid's CTAs leave
  // (one CTA per SM, so every CTA of this grid is running by now); it reads nothing before
  // this grid has completed.
  grid_launch_dependents();
  if (VARLEN && threadIdx.x == 0)
    for (int k = 0; k < NSTAGE && k < my_blocks; ++k) issue(k);


  // Wait for block k in its stage.  The barrier alone tells phases apart only by parity: a group
  // that runs ahead could find the stage still holding block k - 2 NSTAGE's completed phase,
  // of the same parity, while block k - NSTAGE has not been taken out yet.  So the stage's
  // published block number (acquire) must be k first; then the phase test can only see block
  // k's own phase, complete or not.
  auto wait_block = [&](int k) -> bool {
    const int s = k % NSTAGE;
    const uint32_t bar = bar0 + 8u * s, par = (k / NSTAGE) & 1;
    const long long t0 = clock64();
    while (true) {
      if (ld_acquire_shared(gen0 + 4u * s) == k && mbar_try_wait(bar, par)) return true;
      if (*abort_flag) return false;
      if (clock64() - t0 > p.spin_limit) {
        *abort_flag = 1;
        if (atomicCAS(p.err_word, 0, 4 /* ATTN_ERR_TIMEOUT */) == 0) atomicExch(p.err_info, 10);
        return false;
      }
    }
  };

  int n_stores = 0;                  // lane 0: tensor stores this warp has issued from its rows of the buffer
  for (int k = g, it = 0; k < my_blocks; k += C::G, ++it) {
    // Blocks are numbered head-fastest: the groups running at one time read all heads of the
    // same tokens, i.e. contiguous memory.
    const int bt = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
    const int tsr = QKV ? bt / nb1 : 0, bi = bt - tsr * nb1;
    const int h = bi % p.H, blk = (bi / p.H) % p.nblk, b = bi / (p.H * p.nblk);
    const int hb = b * p.H + h;
    // whether this block is rotated (the same for the whole group: a uniform branch)
    const bool rot = ROTATE && (!QKV || tsr < p.rot_tensors);
    const int stage = k % NSTAGE;
    const uint32_t st = base_u32 + stage * C::STAGE_BYTES;
    const bool ok = wait_block(k);
    int tok0 = blk * QROWS, rows = QROWS;
    if constexpr (VARLEN) {
      const int2 inf = stage_info[stage];
      tok0 = inf.x;
      rows = inf.y;
      if (rows == 0) {
        // nothing at this index: pass the stage on once every thread has read its info
        if (group_bar_or(gbar, C::GTHREADS, !ok)) break;
        if (leader && k + NSTAGE < my_blocks) issue(k + NSTAGE);
        continue;
      }
    }

    float v[VPT];
#pragma unroll
    for (int c = 0; c < NW; ++c) {
      const int idx = part * VPT + 8 * c;                  // first element of the chunk
      const int pn = idx / 64, cc = (idx % 64) / 8;        // panel, 16-byte chunk in the row
      const uint32_t addr = st + pn * C::PANEL_BYTES + r * 128 + ((cc ^ (r & 7)) << 4);
      uint32_t w[4];
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(addr));
      if (ROTATE && !ROPE && rot) {
        const uint4 sm = reinterpret_cast<const uint4*>(sign_mask)[idx / 8];
        w[0] ^= sm.x; w[1] ^= sm.y; w[2] ^= sm.z; w[3] ^= sm.w;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[8 * c + 2 * q] = __uint_as_float(w[q] << 16);
        v[8 * c + 2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
      }
    }

    if (VARLEN && r >= rows) {        // the next sequence's row (or past the end): not this block's
#pragma unroll
      for (int e = 0; e < VPT; ++e) v[e] = 0.f;
    }

    if (ROPE) {
      const uint32_t crow = st + C::COARSE_OFF + (r >> 4) * C::TROW + part * C::SEG_BYTES;
      const uint32_t frow = base_u32 + C::OFF_FINE + (r & 15) * C::TROW + part * C::SEG_BYTES;
#pragma unroll
      for (int j = 0; j < VPT / 2; j += 2) {               // two pairs per 16-byte read
        const float4 a = lds128(crow + 8 * j), f = lds128(frow + 8 * j);
        rotary_pair(v[2 * j], v[2 * j + 1], a.x, a.y, f.x, f.y);
        rotary_pair(v[2 * j + 2], v[2 * j + 3], a.z, a.w, f.z, f.w);
      }
    }

    // This warp has read what it needs of the stage.  The group's last warp to get here refills
    // the stage with the block NSTAGE blocks on, while this one is transformed; no warp waits.
    // (A warp whose wait failed does not count: the stage then never refills, later waits run
    // out, and the group stops together at its next barrier.)
    if (__all_sync(0xffffffffu, ok)) {
      if (lane == 0 && atom_add_acq_rel_shared(smem_u32(taken + stage), 1u) % C::GWARPS == C::GWARPS - 1 &&
          k + NSTAGE < my_blocks)
        issue(k + NSTAGE);
    }

    if (ROPE && ROTATE) {
#pragma unroll
      for (int j = 0; j < VPT / 2; j += 4) {
        const uint4 sm = reinterpret_cast<const uint4*>(sign_mask)[(part * VPT / 2 + j) / 4];
        v[2 * j + 1] = __uint_as_float(__float_as_uint(v[2 * j + 1]) ^ sm.x);
        v[2 * j + 3] = __uint_as_float(__float_as_uint(v[2 * j + 3]) ^ sm.y);
        v[2 * j + 5] = __uint_as_float(__float_as_uint(v[2 * j + 5]) ^ sm.z);
        v[2 * j + 7] = __uint_as_float(__float_as_uint(v[2 * j + 7]) ^ sm.w);
      }
    }

    if (ROTATE && rot) {
      // butterflies over the index bits held by this thread: bit 0 pairs the two halves of a
      // packed pair, every higher bit pairs whole pairs, done with f32x2 add/sub
#pragma unroll
      for (int e = 0; e < VPT; e += 2) {
        const float a = v[e], c2 = v[e + 1];
        v[e] = a + c2;
        v[e + 1] = a - c2;
      }
#pragma unroll
      for (int hs = 2; hs < VPT; hs <<= 1)
#pragma unroll
        for (int e = 0; e < VPT; e += 2)
          if ((e & hs) == 0) {
            const uint64_t a2 = f2_pack(v[e], v[e + 1]), b2 = f2_pack(v[e + hs], v[e + hs + 1]);
            f2_unpack(f2_add(a2, b2), v[e], v[e + 1]);
            f2_unpack(f2_sub(a2, b2), v[e + hs], v[e + hs + 1]);
          }
      // the index bits above VPT live in the lanes RPW, 2 RPW apart: the lower part keeps
      // a + b, the upper part a - b
#pragma unroll
      for (int pb = 1; pb < C::TPR; pb <<= 1) {
        const float sgn = (part & pb) ? -1.f : 1.f;
#pragma unroll
        for (int e = 0; e < VPT; e += 2) {
          const float o0 = __shfl_xor_sync(0xffffffffu, v[e], pb * C::RPW);
          const float o1 = __shfl_xor_sync(0xffffffffu, v[e + 1], pb * C::RPW);
          const uint64_t r2 = f2_fma(f2_pack(v[e], v[e + 1]), f2_pack(sgn, sgn), f2_pack(o0, o1));
          f2_unpack(r2, v[e], v[e + 1]);
        }
      }
    }

    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < VPT; e += 2) amax = max3(amax, fabsf(v[e]), fabsf(v[e + 1]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    float* wm = warp_max + C::GWARPS * (it & 1);
    if (lane == 0) wm[gwarp] = amax;
    // the block's one group-wide step: the maximum over its rows (and whether any wait failed)
    if (group_bar_or(gbar, C::GTHREADS, !ok)) break;
    amax = wm[0];
#pragma unroll
    for (int w = 1; w < C::GWARPS; ++w) amax = fmaxf(amax, wm[w]);

    const float inv = amax > 0.f ? 448.f / amax : 0.f;
    if (leader) {
      const float norm = rot ? rsqrtf(static_cast<float>(D)) : 1.f;
      float* sc = !QKV ? p.scale : (tsr == 0 ? p.scale : (tsr == 1 ? p.scale1 : p.scale2));
      sc[static_cast<size_t>(hb) * p.nblk + blk] = amax > 0.f ? (amax * norm) / 448.f : 1.f;
    }
    // Codes into the group's buffer in the output map's swizzled layout, then one tensor store
    // per panel of this warp's rows: whole 128-byte lines reach L2 instead of 16-byte pieces of
    // 32-byte sectors, and rows beyond S are clipped by the store.  The warp's rows of the
    // buffer are free once its previous store has read them.
    if (lane == 0 && n_stores > 0) bulk_wait_read_all();
    __syncwarp();
    {
      const uint64_t inv2 = f2_pack(inv, inv);
#pragma unroll
      for (int c = 0; c < VPT / 16; ++c) {
        uint32_t wq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float y[4];
#pragma unroll
          for (int e = 0; e < 4; e += 2)
            f2_unpack(f2_mul(f2_pack(v[16 * c + 4 * q + e], v[16 * c + 4 * q + e + 1]), inv2), y[e], y[e + 1]);
          wq[q] = pack_e4m3x4(y[0], y[1], y[2], y[3]);
        }
        const int idx = part * VPT + 16 * c;                          // byte in the code row
        if (VARLEN && rows < QROWS) {
          // a partial block: the row straight to global memory, rows past the sequence not at all
          if (r < rows)
            *reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) +
                                      (static_cast<size_t>(tok0 + r) * p.H + h) * D + idx) =
                make_uint4(wq[0], wq[1], wq[2], wq[3]);
          continue;
        }
        const int pn = idx / C::CODE_PANEL, cc = (idx % C::CODE_PANEL) / 16;
        const int sw = C::CODE_PANEL == 128 ? (r & 7) : ((r >> 1) & 3);
        const uint32_t addr = outbuf + pn * (QROWS * C::CODE_PANEL) + r * C::CODE_PANEL + ((cc ^ sw) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(wq[0]), "r"(wq[1]),
                     "r"(wq[2]), "r"(wq[3])
                     : "memory");
      }
    }
    if (!VARLEN || rows == QROWS) {
      fence_proxy_async_smem();
      __syncwarp();
      const int row0 = C::RPW * gwarp;              // this warp's first row of the block
      if (lane == 0 && tok0 + row0 < p.S) {
#pragma unroll
        for (int pn = 0; pn < C::NCPANEL; ++pn)
          tma_store_4d(&m.out[tsr], outbuf + pn * (QROWS * C::CODE_PANEL) + row0 * C::CODE_PANEL, pn * C::CODE_PANEL,
                       h, tok0 + row0, b);
        bulk_commit_group();
        ++n_stores;
      }
    }
  }
  if (lane == 0) bulk_wait_all();
  __syncthreads();

  // On an abort, copies still in flight must land before the CTA exits.
  if (threadIdx.x == 0 && *abort_flag) {
    for (int s = 0; s < NSTAGE; ++s) {
      const int n = issued[s];
      if (n > 0) {
        const long long t0 = clock64();
        while (!mbar_try_wait(bar0 + 8u * s, (n - 1) & 1))
          if (clock64() - t0 > p.spin_limit) break;
      }
    }
  }
}

template <int D, bool ROTATE, bool ROPE, bool VARLEN = false, bool QKV = false>
cudaError_t launch_variant(const QuantMaps& m, const QuantParams& p, int sm_count, cudaStream_t stream) {
  using C = QCfg<D, ROPE, ROTATE, VARLEN>;
  const long long nblocks = static_cast<long long>(p.nblk) * p.H * p.B * (QKV ? 3 : 1);
  // one CTA per SM (a small problem spreads over as many SMs as it has blocks; groups without
  // a block idle)
  const unsigned grid = static_cast<unsigned>(nblocks < sm_count ? nblocks : sm_count);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, hadamard_quant_kernel<D, ROTATE, ROPE, VARLEN, QKV>, m, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D, bool ROTATE, bool ROPE, bool VARLEN = false, bool QKV = false>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(hadamard_quant_kernel<D, ROTATE, ROPE, VARLEN, QKV>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, QCfg<D, ROPE, ROTATE, VARLEN>::SMEM_BYTES);
}

}  // namespace

template <int D>
cudaError_t launch_hadamard_quant(const QuantMaps& m, const QuantParams& p, cudaStream_t stream) {
  static std::atomic<unsigned long long> configured{0};
  static int sm_count[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if ((configured.load() & bit) == 0) {
    if ((e = set_smem<D, true, false>()) != cudaSuccess) return e;
    if ((e = set_smem<D, false, false>()) != cudaSuccess) return e;
    if ((e = set_smem<D, true, true>()) != cudaSuccess) return e;
    if ((e = set_smem<D, false, true>()) != cudaSuccess) return e;
    if ((e = set_smem<D, true, false, true>()) != cudaSuccess) return e;
    if ((e = set_smem<D, false, false, true>()) != cudaSuccess) return e;
    if ((e = set_smem<D, true, true, true>()) != cudaSuccess) return e;
    if ((e = set_smem<D, false, true, true>()) != cudaSuccess) return e;
    if ((e = set_smem<D, true, false, false, true>()) != cudaSuccess) return e;
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sm_count[dev & 63] = n;
    configured.fetch_or(bit);
  }
  const int sms = sm_count[dev & 63];
  const bool rot = p.signs != nullptr, rope = p.rope_cs != nullptr;
  if (p.n_tensors == 3) return launch_variant<D, true, false, false, true>(m, p, sms, stream);
  if (p.cu_seqlens != nullptr) {
    if (rope)
      return rot ? launch_variant<D, true, true, true>(m, p, sms, stream)
                 : launch_variant<D, false, true, true>(m, p, sms, stream);
    return rot ? launch_variant<D, true, false, true>(m, p, sms, stream)
               : launch_variant<D, false, false, true>(m, p, sms, stream);
  }
  if (rope)
    return rot ? launch_variant<D, true, true>(m, p, sms, stream)
               : launch_variant<D, false, true>(m, p, sms, stream);
  return rot ? launch_variant<D, true, false>(m, p, sms, stream)
             : launch_variant<D, false, false>(m, p, sms, stream);
}

template cudaError_t launch_hadamard_quant<64>(const QuantMaps&, const QuantParams&, cudaStream_t);
template cudaError_t launch_hadamard_quant<128>(const QuantMaps&, const QuantParams&, cudaStream_t);
template cudaError_t launch_hadamard_quant<256>(const QuantMaps&, const QuantParams&, cudaStream_t);

}  // namespace ea46
