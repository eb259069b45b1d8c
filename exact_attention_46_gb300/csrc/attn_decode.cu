// attn_decode.cu -- attention for few query tokens against many keys (decoding), with grouped
// key/value heads, for sm_103a.
//
// What it computes (readings; the hada.io FA3 summary, "Weitere Optimierungen und künftige
// Integration", names LLM inference as future work and defines nothing): Q [B, Sq, Hq, D]
// against K, V [B, Sk, Hkv, D], Hq = G * Hkv, query head h reading key/value head h / G;
// under the causal mask query i sees keys j <= Sk - Sq + i (the queries are the last Sq
// positions).  O [B, Sq, Hq, D] bf16, lse [B, Hq, Sq] fp32.
//
// Design: with Sq * G query rows per key/value head the work is a stream over K and V --
// bandwidth-bound -- so the kernel's job is to keep HBM busy:
//   * one CTA per (b, key/value head, key split); its G heads x Sq tokens are packed into the
//     rows of one 128-row tcgen05 tile (row r = token r / G, head r % G) by a 5-D TMA box, so
//     every K/V tile is read once for the whole group;
//   * the keys are split over as many CTAs as fill the GPU (B * Hkv alone is often < 152);
//     each split writes its normalised partial O and lse to a caller workspace and a combine
//     kernel merges them (lse = log sum exp lse_c, O = sum exp(lse_c - lse) O_c); with one
//     split the kernel writes O and lse itself;
//   * a load warp streams K_j, V_j through a ring of shared-memory slots; one thread issues
//     S = Q K_j^T and O += P V_j on the tensor core; softmax warps (thread = tile row) run the
//     online softmax as the prefill kernel does (lazy rescale, P in Tensor Memory);
//   * with few query rows (R = G * Sq) the softmax of a tile is R rows' passes over 128 keys,
//     one thread per row, and a warp may only reach the Tensor Memory lanes of its own quarter
//     -- its own SM sub-partition, with its own exp2 unit.  So the R rows are copied REP
//     times into the tile (REP = 4 for R <= 32, 2 for R <= 64, else 1; one more TMA box per
//     copy), copy c takes keys [c * 128 / REP, (c + 1) * 128 / REP) of every tile, and the
//     four sub-partitions share the work.  Per tile the copies exchange their row maxima
//     (shared memory and a named barrier); each keeps its own row sum and partial O, written
//     into its own P buffer in Tensor Memory (zero outside its keys), and the epilogue adds
//     the copies' O and sums through shared memory;
//   * FP8 (E4M3 Q, K, V with the quantiser's block scales): the same kernel on kind::f8f6f4;
//     a row's query scale and a tile's key scale multiply the logit constant, the tile's value
//     scale enters the exponent as log2(sv_j / max sv) and the epilogue as max sv (the maximum
//     over the split's tiles), as in the prefill kernel.
// A split may see no key of a row under the causal mask; its partial then carries lse = -inf
// and weight zero.  Every mbarrier wait is bounded.
#include <atomic>
#include <cfloat>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ea46 {

namespace {

constexpr float TAU_DEC = 8.0f;
constexpr float LN2_DEC = 0.69314718055994530942f;

template <int D, bool FP8>
struct DecCfg {
  static constexpr int ESZ = FP8 ? 1 : 2;
  static constexpr int ROW_BYTES = D * ESZ;
  static constexpr int PANEL_ROW = ROW_BYTES >= 128 ? 128 : ROW_BYTES;  // swizzle span
  static constexpr int NPANEL = ROW_BYTES / PANEL_ROW;
  static constexpr int PANEL_ELEMS = PANEL_ROW / ESZ;
  static constexpr int PANEL_BYTES = 128 * PANEL_ROW;
  static constexpr int TILE_BYTES = 128 * ROW_BYTES;
  static constexpr int NSLOT = ROW_BYTES == 256 ? 6 : (ROW_BYTES == 128 ? 12 : 16);   // K/V tiles in flight
  static constexpr uint32_t SBO = 8 * PANEL_ROW;
  static constexpr uint32_t LAYOUT = PANEL_ROW == 128 ? 2u : 4u;          // SW128 / SW64
  static constexpr int KSTEPS_QK = ROW_BYTES / 32;
  static constexpr int STEPS_PER_PANEL = PANEL_ROW / 32;
  static constexpr int UMMA_K = FP8 ? 32 : 16;
  static constexpr int KSTEPS_PV = 128 / UMMA_K;
  static constexpr uint32_t FMT = FP8 ? 0u : 1u;                           // E4M3 / BF16
  static constexpr uint32_t IDESC_QK = instr_desc(FMT, 0, 128, 128);
  static constexpr uint32_t IDESC_PV = instr_desc(FMT, 1, 128, D);
  // Tensor Memory: S buffers at columns 0 and 128, O at 256, two P buffers after O
  static constexpr uint32_t O_COL = 256, P_COL = 256 + D;
  static constexpr uint32_t PW = FP8 ? 32 : 64;                            // columns of P (128 keys)
  static constexpr int NBAR = 8 + 2 * NSLOT;
  // per-row exchange between replicas: [2][128] floats, then failure flags [2]
  static constexpr int RED_BYTES = 2 * 128 * 4 + 16;
  static constexpr int SMEM_BYTES = 1024 + (1 + NSLOT) * TILE_BYTES + NBAR * 8 + 16 + RED_BYTES;
  static constexpr int THREADS = 32 * 6;
  static constexpr int LOAD_WARP = 4, MMA_WARP = 5;
  static constexpr int OBUF_STRIDE = D + 4;     // floats per row of the epilogue's partial-O buffer
  static_assert(D == 64 || D == 128, "head dimension");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(P_COL + 2 * PW <= 512, "Tensor Memory budget");
  static_assert(128 * OBUF_STRIDE * 4 <= NSLOT * TILE_BYTES, "partial-O buffer fits the K/V ring");
};

enum : int { WHERE_DEC_LOAD = 21, WHERE_DEC_MMA = 22, WHERE_DEC_SOFTMAX = 23 };

__device__ __forceinline__ void wait_drain_dec(uint32_t bar, uint32_t parity, long long limit) {
  if (mbar_try_wait(bar, parity)) return;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > limit) return;
}

// REP: copies of the R packed query rows in the 128-row tile (R <= 128 / REP); copy c takes
// keys [c * 128 / REP, (c + 1) * 128 / REP) of every tile.
template <int D, bool FP8, bool CAUSAL, int REP>
__global__ void __launch_bounds__(DecCfg<D, FP8>::THREADS, 1)
    attn_decode_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
  using C = DecCfg<D, FP8>;
  constexpr int NSLOT = C::NSLOT;
  constexpr int RROWS = 128 / REP;           // tile rows (lanes) of one copy
  constexpr int CW = 128 / REP;              // keys of a tile one copy takes
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const uint32_t sQ = base_u32;
  const uint32_t sKV = base_u32 + C::TILE_BYTES;
  const uint32_t bar0 = sKV + NSLOT * C::TILE_BYTES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + (bar0 - base_u32) + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(tmem_slot + 4);                   // [2][128]
  volatile int* qfail = reinterpret_cast<volatile int*>(red + 2 * 128);   // [2]
  const uint32_t BAR_Q = bar0, BAR_O = bar0 + 8, BAR_DONE = bar0 + 16, BAR_PV = bar0 + 24;
  auto BAR_S = [&](int b2) { return bar0 + 32 + 8u * b2; };       // S buffer b2 written
  auto BAR_P = [&](int b2) { return bar0 + 48 + 8u * b2; };       // P buffer b2 written
  auto BAR_FULL = [&](int s) { return bar0 + 64 + 8u * s; };
  auto BAR_EMPTY = [&](int s) { return bar0 + 64 + 8u * (NSLOT + s); };

  const uint32_t warp = warp_id(), lane = lane_id();
  // CTA -> (split, b, key/value head)
  const int bkv = static_cast<int>(blockIdx.x) % (p.B * p.Hkv);
  const int split = static_cast<int>(blockIdx.x) / (p.B * p.Hkv);
  const int b = bkv / p.Hkv, hkv = bkv % p.Hkv;
  const int nk = (p.Sk + 127) / 128;
  const int t0 = split * p.tiles_per_split;
  const int t1 = t0 + p.tiles_per_split < nk ? t0 + p.tiles_per_split : nk;
  const int ntile = t1 - t0;                 // >= 1 (the host never forms an empty split)
  const int R = p.G * p.Sq;                  // packed query rows (<= RROWS)

  if (threadIdx.x == 0) {
    mbar_init(BAR_Q, 1);
    mbar_init(BAR_O, 1);
    mbar_init(BAR_DONE, 1);
    mbar_init(BAR_PV, 1);
    for (int b2 = 0; b2 < 2; ++b2) {
      mbar_init(BAR_S(b2), 1);
      mbar_init(BAR_P(b2), 4);
    }
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(BAR_FULL(s), 1);
      mbar_init(BAR_EMPTY(s), 1);
    }
    *abort_flag = 0;
    qfail[0] = 0;
    qfail[1] = 0;
    fence_barrier_init();
  }
  if (warp == C::MMA_WARP) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{p.spin_limit, abort_flag, p.err_word, p.err_info};

  if (warp == C::LOAD_WARP) {
    if (lane == 0) {
      const uint64_t pol_q = l2_policy_evict_first(), pol_kv = l2_policy_evict_first();
      mbar_arrive_expect_tx(BAR_Q, REP * C::NPANEL * R * C::PANEL_ROW);
      for (int c = 0; c < REP; ++c)
        for (int pn = 0; pn < C::NPANEL; ++pn)
          tma_load_5d(sQ + pn * C::PANEL_BYTES + c * RROWS * C::PANEL_ROW, &tmQ, BAR_Q, pn * C::PANEL_ELEMS, 0,
                      hkv, 0, b, pol_q);
      int issued = 0;
      for (int j = 0; j < ntile && !*abort_flag; ++j) {
        for (int kind = 0; kind < 2; ++kind) {
          const int slot = issued % NSLOT;
          if (!wait_bounded(BAR_EMPTY(slot), ((issued / NSLOT) & 1) ^ 1u, ctl, WHERE_DEC_LOAD)) break;
          mbar_arrive_expect_tx(BAR_FULL(slot), C::TILE_BYTES);
          const CUtensorMap* m = kind == 0 ? &tmK : &tmV;
          for (int pn = 0; pn < C::NPANEL; ++pn)
            tma_load_4d(sKV + slot * C::TILE_BYTES + pn * C::PANEL_BYTES, m, BAR_FULL(slot), pn * C::PANEL_ELEMS,
                        hkv, 128 * (t0 + j), b, pol_kv);
          ++issued;
        }
      }
      if (*abort_flag) {
        wait_drain_dec(BAR_Q, 0, p.spin_limit);
        for (int i = (issued > NSLOT ? issued - NSLOT : 0); i < issued; ++i)
          wait_drain_dec(BAR_FULL(i % NSLOT), (i / NSLOT) & 1, p.spin_limit);
      }
    }
  } else if (warp == C::MMA_WARP) {
    if (lane == 0) {
      const uint64_t dq = smem_desc(sQ, 16, C::SBO, C::LAYOUT);
      const uint64_t dk0 = smem_desc(sKV, 16, C::SBO, C::LAYOUT);
      const uint64_t dv0 = smem_desc(sKV, C::PANEL_BYTES, C::SBO, C::LAYOUT);
      bool ok = wait_bounded(BAR_Q, 0, ctl, WHERE_DEC_MMA);
      // ring position of K_j is 2j, of V_j 2j + 1 (the load order)
      auto qk = [&](int j) -> bool {
        const int idx = 2 * j, ks = idx % NSLOT;
        if (!wait_bounded(BAR_FULL(ks), (idx / NSLOT) & 1, ctl, WHERE_DEC_MMA)) return false;
        tc_fence_after();
        const uint64_t bk = dk0 + ((ks * C::TILE_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS_QK; ++kk) {
          const uint32_t off = ((kk / C::STEPS_PER_PANEL) * C::PANEL_BYTES + (kk % C::STEPS_PER_PANEL) * 32) >> 4;
          if (FP8) mma_f8_ss(tmem + 128u * (j & 1), dq + off, bk + off, C::IDESC_QK, kk > 0);
          else     mma_f16_ss(tmem + 128u * (j & 1), dq + off, bk + off, C::IDESC_QK, kk > 0);
        }
        mma_commit(BAR_S(j & 1));
        mma_commit(BAR_EMPTY(ks));
        return true;
      };
      if (ok) ok = qk(0);
      for (int j = 0; ok && j < ntile; ++j) {
        // S(j+1) overwrites S(j-1), which the softmax read before it handed over P(j-1)
        if (j + 1 < ntile && !(ok = qk(j + 1))) break;
        if (!(ok = wait_bounded(BAR_P(j & 1), (j >> 1) & 1, ctl, WHERE_DEC_MMA))) break;
        const int idx = 2 * j + 1, vs = idx % NSLOT;
        if (!(ok = wait_bounded(BAR_FULL(vs), (idx / NSLOT) & 1, ctl, WHERE_DEC_MMA))) break;
        tc_fence_after();
        const uint64_t bv = dv0 + ((vs * C::TILE_BYTES) >> 4);
        const uint32_t pa = tmem + C::P_COL + C::PW * (j & 1);
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS_PV; ++kk) {
          const uint32_t off = (kk * C::UMMA_K * C::PANEL_ROW) >> 4;
          if (FP8) mma_f8_ts(tmem + C::O_COL, pa + 8u * kk, bv + off, C::IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
          else     mma_f16_ts(tmem + C::O_COL, pa + 8u * kk, bv + off, C::IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(BAR_PV);
        mma_commit(BAR_EMPTY(vs));
      }
      if (ok) mma_commit(BAR_O);
      mma_commit(BAR_DONE);
      wait_drain_dec(BAR_DONE, 0, p.spin_limit);
    }
  } else {
    // softmax warps 0..3: thread t = tile row (lane) t; copy c = t / RROWS of packed row
    // r = t % RROWS = (token r / G, head r % G), which takes keys [c * CW, (c + 1) * CW)
    const int t = static_cast<int>(threadIdx.x);
    const int c = t / RROWS, r = t % RROWS;
    const uint32_t tl = tmem + ((warp * 32u) << 16);
    const int tok = r / p.G;
    const int lim_all = p.Sk - p.Sq + tok;    // last visible key under the mask
    float m_run = -INFINITY, l_run = 0.f;     // l_run: this copy's keys only
    // FP8: this row's query scale, and the largest value scale of the split's key tiles
    float cq = p.c_log2, sv_max = 1.f;
    const size_t kv_blk = (static_cast<size_t>(b) * p.Hkv + hkv) * p.nkb;
    if (FP8) {
      if (r < R && p.q_scale != nullptr)
        cq *= p.q_scale[(static_cast<size_t>(b) * p.Hq + hkv * p.G + r % p.G) * p.nqb + tok / 128];
      if (p.v_scale != nullptr) {
        sv_max = 0.f;
        for (int jj = static_cast<int>(lane); jj < ntile; jj += 32) sv_max = fmaxf(sv_max, p.v_scale[kv_blk + t0 + jj]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sv_max = fmaxf(sv_max, __shfl_xor_sync(0xffffffffu, sv_max, o));
        sv_max = fmaxf(sv_max, 0x1p-96f);  // every value scale 0: O = 0, l still counts
      }
    }
    if constexpr (REP > 1) {
      // P columns outside this copy's keys stay zero: clear both P buffers once
      uint32_t z[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = 0u;
#pragma unroll
      for (uint32_t col = 0; col < 2 * C::PW; col += 32) tmem_st32(tl + C::P_COL + col, z);
    }
    // Max (or sum) of v over the copies of row r, through red[buf].  The named barrier over the
    // four softmax warps also orders every copy's S loads before any P store.  It cannot time
    // out, so the warps leave the loop only together: a warp whose bounded wait gave up
    // ("bad") raises qfail[buf] and still comes to the barrier; after it every warp reads the
    // flag and all stop, or none does.  A failure found after the barrier of tile j goes into
    // the flag read at the next one.
    bool bad = false;
    auto copies_reduce = [&](float v, int buf, bool is_max, bool& failed) -> float {
      if constexpr (REP == 1) {
        failed = bad;
        return v;
      } else {
        float* rb = red + buf * 128;
        rb[t] = v;
        if (bad) qfail[buf] = 1;
        tc_fence_before();
        named_bar_sync(1u, 128u);
        tc_fence_after();
        failed = qfail[buf] != 0;
        float x = rb[r];
#pragma unroll
        for (int cc = 1; cc < REP; ++cc) x = is_max ? fmaxf(x, rb[cc * RROWS + r]) : x + rb[cc * RROWS + r];
        return x;
      }
    };
    // FP8: the key and value scales of the split's tiles, 32 tiles at a time in the lanes'
    // registers (lane i: tile 32 * n + i), the next 32 fetched a batch ahead, so that no global
    // load sits between one tile's P hand-off and the next tile's S
    float sk_cur = 1.f, sv_cur = 1.f, sk_nxt = 1.f, sv_nxt = 1.f;
    auto fetch_scales = [&](int j0, float& skr, float& svr) {
      const int jj = j0 + static_cast<int>(lane);
      skr = (p.k_scale != nullptr && jj < ntile) ? p.k_scale[kv_blk + t0 + jj] : 1.f;
      svr = (p.v_scale != nullptr && jj < ntile) ? p.v_scale[kv_blk + t0 + jj] : 1.f;
    };
    if (FP8) {
      fetch_scales(0, sk_cur, sv_cur);
      fetch_scales(32, sk_nxt, sv_nxt);
    }
    for (int j = 0; j < ntile; ++j) {
      const int kb = 128 * (t0 + j);
      float cmul = p.c_log2, bias = 0.f, inv_r = 1.f;
      if (FP8) {
        if (j > 0 && (j & 31) == 0) {
          sk_cur = sk_nxt;
          sv_cur = sv_nxt;
          fetch_scales(j + 32, sk_nxt, sv_nxt);
        }
        const float sk = __shfl_sync(0xffffffffu, sk_cur, j & 31);
        const float sv_raw = __shfl_sync(0xffffffffu, sv_cur, j & 31);
        // a zero scale (a block of zeros) as 2^-30 of the largest: its numerators vanish in E4M3,
        // the row sum still takes them at full weight
        const float sv = fmaxf(sv_raw, sv_max * 0x1p-30f);
        cmul = cq * sk;
        bias = __log2f(sv / sv_max);
        inv_r = sv_max / sv;
      }
      const uint32_t sb = tl + 128u * (j & 1) + c * CW;
      if (!bad && !warp_wait(BAR_S(j & 1), (j >> 1) & 1, ctl, WHERE_DEC_SOFTMAX)) bad = true;
      uint32_t sr[CW / 32][32];
      if (!bad) {
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < CW / 32; ++q) tmem_ld32(sb + 32u * q, sr[q]);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int q = 0; q < CW / 32; ++q)
#pragma unroll
          for (int i = 0; i < 32; ++i) sr[q][i] = __float_as_uint(-INFINITY);
      }
#pragma unroll
      for (int q = 0; q < CW / 32; ++q)
#pragma unroll
        for (int i = 0; i < 32; ++i) reg_fence(sr[q][i]);
      // visible keys of this copy's slice: kb + c * CW + col <= lim (lim < 0: none).  Rows past
      // the R packed query rows hold whatever shared memory held (the TMA boxes write R rows
      // per copy): they see no key, so they never ask for a rescale of O
      const int lim = r < R ? (CAUSAL ? (lim_all < p.Sk - 1 ? lim_all : p.Sk - 1) : p.Sk - 1) - kb - c * CW : -1;
      if (lim < CW - 1) {
#pragma unroll
        for (int q = 0; q < CW / 32; ++q)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * q + i > lim) sr[q][i] = __float_as_uint(-INFINITY);
      }
      float mt = -INFINITY;
#pragma unroll
      for (int q = 0; q < CW / 32; ++q)
#pragma unroll
        for (int i = 0; i < 32; i += 2) mt = max3(mt, __uint_as_float(sr[q][i]), __uint_as_float(sr[q][i + 1]));
      bool failed = false;
      mt = copies_reduce(mt, j & 1, true, failed) * cmul;
      if (failed) {                           // every softmax warp stops here
        bad = true;
        break;
      }
      bool rescale = false;
      float alpha = 1.f;
      if (mt > m_run + TAU_DEC || (m_run == -INFINITY && mt != -INFINITY)) {
        alpha = m_run == -INFINITY ? 0.f : ex2(m_run - mt);
        m_run = mt;
        l_run *= alpha;
        rescale = j > 0;
      }
      const float off = (m_run == -INFINITY ? 0.f : m_run) - bias;   // no visible key yet: p = 0
      const uint32_t pb = tl + C::P_COL + C::PW * (j & 1);
      float ls = 0.f;
#pragma unroll
      for (int q = 0; q < CW / 32; ++q) {
        if constexpr (!FP8) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float p0 = ex2(fmaf(__uint_as_float(sr[q][2 * i]), cmul, -off));
            const float p1 = ex2(fmaf(__uint_as_float(sr[q][2 * i + 1]), cmul, -off));
            ls += p0 + p1;
            pk[i] = pack_bf16x2(p0, p1);
          }
          tmem_st16(pb + c * (CW / 2) + 16u * q, pk);
        } else {
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float pv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              pv[e] = ex2(fmaf(__uint_as_float(sr[q][4 * i + e]), cmul, -off));
              ls += pv[e];
            }
            pk[i] = pack_e4m3x4(pv[0], pv[1], pv[2], pv[3]);
          }
          tmem_st8(pb + c * (CW / 4) + 8u * q, pk);
        }
      }
      l_run += ls * inv_r;
      if (__any_sync(0xffffffffu, rescale)) {
        // O must hold PV(j-1) complete (PV(j) waits for this warp's arrival below); S(j) may
        // have been issued before PV(j-1), so wait for PV(j-1)'s completion explicitly
        if (!warp_wait(BAR_PV, (j - 1) & 1, ctl, WHERE_DEC_SOFTMAX)) {
          bad = true;                         // reported at the next exchange
          if (REP == 1) break;
          continue;
        }
        tc_fence_after();
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          uint32_t o[32];
          tmem_ld32(tl + C::O_COL + 32u * q, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            reg_fence(o[i]);
            o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          }
          tmem_st32(tl + C::O_COL + 32u * q, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR_P(j & 1));
    }
    // every softmax warp comes here having run the loop as far as the others; the row sums of
    // the copies are exchanged (with the failure flag) whatever happened
    if (!bad && !warp_wait(BAR_O, 0, ctl, WHERE_DEC_SOFTMAX)) bad = true;
    bool failed = false;
    l_run = copies_reduce(l_run, ntile & 1, false, failed);
    if (!failed) {
      tc_fence_after();
      const bool valid = r < R;
      const int g = r % p.G, h = hkv * p.G + g;
      const float inv_l = l_run > 0.f ? sv_max / l_run : 0.f;
      const float lse = l_run > 0.f ? (m_run + __log2f(l_run)) * LN2_DEC : -INFINITY;
      const size_t row = (static_cast<size_t>(b) * p.Hq + h) * p.Sq + (valid ? tok : 0);   // [B, Hq, Sq]
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + ((static_cast<size_t>(b) * p.Sq + tok) * p.Hq + h) * D;
      float* wrow = p.n_split > 1 ? p.ws_o + (static_cast<size_t>(split) * p.rows_total + row) * D : nullptr;
      // writes 8 output columns from col: O / l as bf16, or the normalised partial in fp32
      auto put8 = [&](int col, const float* v) {
        if (p.n_split == 1) {
          *reinterpret_cast<uint4*>(orow + col) =
              make_uint4(pack_bf16x2(v[0] * inv_l, v[1] * inv_l), pack_bf16x2(v[2] * inv_l, v[3] * inv_l),
                         pack_bf16x2(v[4] * inv_l, v[5] * inv_l), pack_bf16x2(v[6] * inv_l, v[7] * inv_l));
        } else {
          reinterpret_cast<float4*>(wrow + col)[0] = make_float4(v[0] * inv_l, v[1] * inv_l, v[2] * inv_l, v[3] * inv_l);
          reinterpret_cast<float4*>(wrow + col)[1] = make_float4(v[4] * inv_l, v[5] * inv_l, v[6] * inv_l, v[7] * inv_l);
        }
      };
      if constexpr (REP == 1) {
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          uint32_t o[32];
          tmem_ld32(tl + C::O_COL + 32u * q, o);
          tmem_wait_ld();
          float f[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            reg_fence(o[i]);
            f[i] = __uint_as_float(o[i]);
          }
          if (valid)
#pragma unroll
            for (int v8 = 0; v8 < 4; ++v8) put8(32 * q + 8 * v8, f + 8 * v8);
        }
      } else {
        // the copies' partial O rows meet in shared memory over the K/V ring (every load has
        // landed: the last PV waited for them); copy c then writes columns
        // [c * D / REP, (c + 1) * D / REP) of row r
        float* obuf = reinterpret_cast<float*>(base + (sKV - base_u32));
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          uint32_t o[32];
          tmem_ld32(tl + C::O_COL + 32u * q, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) reg_fence(o[i]);
          float4* dst = reinterpret_cast<float4*>(obuf + t * C::OBUF_STRIDE + 32 * q);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            dst[v4] = make_float4(__uint_as_float(o[4 * v4]), __uint_as_float(o[4 * v4 + 1]),
                                  __uint_as_float(o[4 * v4 + 2]), __uint_as_float(o[4 * v4 + 3]));
        }
        named_bar_sync(1u, 128u);
        if (valid) {
          constexpr int OWR = D / REP;
#pragma unroll 1
          for (int col = c * OWR; col < (c + 1) * OWR; col += 8) {
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
            for (int cc = 0; cc < REP; ++cc) {
              const float4* src = reinterpret_cast<const float4*>(obuf + (cc * RROWS + r) * C::OBUF_STRIDE + col);
              const float4 a = src[0], bq = src[1];
              acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
              acc[4] += bq.x; acc[5] += bq.y; acc[6] += bq.z; acc[7] += bq.w;
            }
            put8(col, acc);
          }
        }
      }
      if (valid && c == 0) {
        if (p.n_split == 1) {
          if (p.lse != nullptr) p.lse[row] = lse;
        } else {
          p.ws_l[static_cast<size_t>(split) * p.rows_total + row] = lse;
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge of the key splits: one warp per (b, h, token) row.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecodeParams p) {
  const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = static_cast<int>(threadIdx.x & 31);
  if (w >= p.rows_total) return;
  const size_t row = static_cast<size_t>(w);            // (b * Hq + h) * Sq + tok
  float mx = -INFINITY;
  for (int c = 0; c < p.n_split; ++c) mx = fmaxf(mx, p.ws_l[static_cast<size_t>(c) * p.rows_total + row]);
  float acc[D / 32];
#pragma unroll
  for (int e = 0; e < D / 32; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  for (int c = 0; c < p.n_split; ++c) {
    const float lc = p.ws_l[static_cast<size_t>(c) * p.rows_total + row];
    const float wgt = lc == -INFINITY ? 0.f : __expf(lc - mx);
    wsum += wgt;
    const float* oc = p.ws_o + (static_cast<size_t>(c) * p.rows_total + row) * D;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) acc[e] = fmaf(wgt, oc[lane + 32 * e], acc[e]);
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const int tok = static_cast<int>(row % p.Sq);
  const int bh = static_cast<int>(row / p.Sq);
  const int b = bh / p.Hq, h = bh % p.Hq;
  __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.o) + ((static_cast<size_t>(b) * p.Sq + tok) * p.Hq + h) * D;
#pragma unroll
  for (int e = 0; e < D / 32; ++e) dst[lane + 32 * e] = __float2bfloat16_rn(acc[e] * inv);
  if (lane == 0 && p.lse != nullptr) p.lse[row] = mx + logf(wsum);
}

template <int D, bool FP8, bool CAUSAL, int REP>
cudaError_t launch_decode_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const DecodeParams& p, cudaStream_t st) {
  using C = DecCfg<D, FP8>;
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if ((configured.load() & bit) == 0) {
    e = cudaFuncSetAttribute(attn_decode_kernel<D, FP8, CAUSAL, REP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  const unsigned grid = static_cast<unsigned>(p.B * p.Hkv * p.n_split);
  attn_decode_kernel<D, FP8, CAUSAL, REP><<<grid, C::THREADS, C::SMEM_BYTES, st>>>(tq, tk, tv, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.n_split > 1) {
    const long long threads = p.rows_total * 32;
    decode_combine_kernel<D><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, st>>>(p);
    e = cudaGetLastError();
  }
  return e;
}

// Copies of the packed query rows: as many as fit the 128-row tile, at most four (one per
// lane quarter, hence per SM sub-partition).
template <int D, bool FP8, bool CAUSAL>
cudaError_t launch_decode_rep(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const DecodeParams& p, cudaStream_t st) {
  const int R = p.G * p.Sq;
  if (R <= 32) return launch_decode_d<D, FP8, CAUSAL, 4>(tq, tk, tv, p, st);
  if (R <= 64) return launch_decode_d<D, FP8, CAUSAL, 2>(tq, tk, tv, p, st);
  return launch_decode_d<D, FP8, CAUSAL, 1>(tq, tk, tv, p, st);
}

}  // namespace

cudaError_t launch_attn_decode(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeParams& p, int D, bool fp8, bool causal, cudaStream_t st) {
  if (fp8) {
    if (D == 64) return causal ? launch_decode_rep<64, true, true>(tq, tk, tv, p, st)
                               : launch_decode_rep<64, true, false>(tq, tk, tv, p, st);
    return causal ? launch_decode_rep<128, true, true>(tq, tk, tv, p, st) : launch_decode_rep<128, true, false>(tq, tk, tv, p, st);
  }
  if (D == 64) return causal ? launch_decode_rep<64, false, true>(tq, tk, tv, p, st)
                             : launch_decode_rep<64, false, false>(tq, tk, tv, p, st);
  return causal ? launch_decode_rep<128, false, true>(tq, tk, tv, p, st) : launch_decode_rep<128, false, false>(tq, tk, tv, p, st);
}

}  // namespace ea46
