// attn_bwd.cu -- backward pass of the fused attention (dQ, dK, dV) for sm_103a.
//
// What it computes: the gradients of O = softmax(scale * Q K^T [causal]) V given dO, from Q, K,
// V, O and the forward's per-row log-sum-exp -- FlashAttention's recomputation (hada.io FA3
// summary, "Rückblick auf den FlashAttention-Ansatz": the score matrix is never stored, what
// the backward needs is recomputed tile by tile).  Per (b, h), with P = exp(scale S - lse):
//   dV = P^T dO,   dP = dO V^T,   Delta_i = sum_d dO_id O_id,   dS = P * (dP - Delta),
//   dQ = scale dS K,   dK = scale dS^T Q.
//
// Three kernels (own design; the pages give no backward schedule):
//   1. delta:  Delta and lse * log2(e) per row into a workspace [B*H][2][S rounded up to 128]
//              (bandwidth-bound, plain loads).
//   2. dK/dV:  CTA = 128 keys of one (b, h); K, V stay in shared memory while Q_j, dO_j and
//              the rows' Delta / lse stream through a TMA ring.  Per query tile the tensor core
//              forms S^T = K Q_j^T and dP^T = V dO_j^T in Tensor Memory; the eight compute
//              warps (thread = key row = TMEM lane; two warps per row, each half the columns)
//              turn them into P^T and dS^T (bf16, written back over S^T and dP^T); then
//              dV += P^T dO_j and dK += dS^T Q_j accumulate in
//              Tensor Memory (A operand from Tensor Memory, B = dO_j / Q_j read N-major).
//   3. dQ:     CTA = 128 queries; Q, dO resident, K_j, V_j stream (rings of their own); S =
//              Q K_j^T (double-buffered in Tensor Memory) and dP = dO V_j^T, dS by the compute
//              warps (thread = query row), dQ += dS K_j; S(j+1) and dP(j+1) are issued before
//              dQ(j), so the compute warps do not wait for the tensor core between tiles.
//   Recomputing S and dP in both kernels costs two extra GEMMs per tile pair but needs no
//   atomics and no fp32 dQ accumulator in device memory.
//
// Grouped-query attention (H query heads over Hkv key/value heads, query head h reading head
// h / (H / Hkv)) is the same computation with each K/V head repeated over its group: dQ is
// unchanged, and dK, dV of a key/value head are the sums over the group's query heads.  The
// dK/dV CTA therefore belongs to (key tile, b, key/value head) and streams the query tiles of
// every head of the group through the same ring, so the sum stays in Tensor Memory.
//
// Tensor Memory (512 columns): S at 0 (P over columns 0-31 and 64-95: each half of the compute
// warps over its own half of S), dP at 128 (dS likewise), then the accumulators (dV, dK at 256
// and 256 + D; dQ at 256, and the dQ kernel's second S buffer at 384).  D = 64 or 128.
//
// Every mbarrier wait is bounded (ptx.cuh); a wait that runs out records ATTN_ERR_TIMEOUT and
// every role leaves through the common exit, which frees Tensor Memory.
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ea46 {

namespace {

constexpr float LOG2E = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int PANEL_ROW = 128;                        // bytes of a row per swizzle panel
  static constexpr int NPANEL = ROW_BYTES / PANEL_ROW;         // 1 (D = 64), 2 (D = 128)
  static constexpr int PANEL_ELEMS = 64;
  static constexpr int PANEL_BYTES = 128 * PANEL_ROW;
  static constexpr int TILE_BYTES = 128 * ROW_BYTES;
  static constexpr int VEC_BYTES = 2 * 128 * 4;                // Delta, lse*log2e of 128 rows
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES + VEC_BYTES;
  static constexpr int NSTAGE = D == 64 ? 4 : 2;
  static constexpr uint32_t SBO = 8 * PANEL_ROW;
  static constexpr uint32_t LAYOUT = 2u;                       // 128-byte swizzle
  static constexpr int KSTEPS_SS = ROW_BYTES / 32;             // 16 bf16 of the reduction per MMA
  static constexpr int STEPS_PER_PANEL = PANEL_ROW / 32;
  static constexpr int KSTEPS_TS = 128 / 16;
  static constexpr uint32_t IDESC_SS = instr_desc(1, 0, 128, 128);
  static constexpr uint32_t IDESC_TS = instr_desc(1, 1, 128, D);
  static constexpr int NBAR = 4 + 2 * NSTAGE + 3;     // ..., done, dP ready, dS ready
  static constexpr int SMEM_BYTES = 1024 + 2 * TILE_BYTES + NSTAGE * STAGE_BYTES + NBAR * 8 + 16;
  // 8 compute warps: two per Tensor-Memory lane quarter, each taking 64 of a tile's 128
  // columns (the compute is elementwise, so the halves never meet), then 1 load, 1 MMA
  static constexpr int COMPUTE_WARPS = 8;
  static constexpr int THREADS = 32 * (COMPUTE_WARPS + 2);
  static constexpr int LOAD_WARP = COMPUTE_WARPS, MMA_WARP = COMPUTE_WARPS + 1;
  static_assert(D == 64 || D == 128, "head dimension");
  static_assert(256 + 2 * D <= 512, "Tensor Memory budget");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

enum : int { WHERE_BWD_LOAD = 11, WHERE_BWD_MMA = 12, WHERE_BWD_COMPUTE = 13 };

__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, long long limit) {
  if (mbar_try_wait(bar, parity)) return;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > limit) return;
}

// ---------------------------------------------------------------- kernel 1: delta --
// ws[(2 bh) * Sp + s] = sum_d dO O, ws[(2 bh + 1) * Sp + s] = lse * log2(e); 0 for s >= S.
template <int D>
__global__ void __launch_bounds__(256) delta_kernel(const __nv_bfloat16* __restrict__ o,
                                                    const __nv_bfloat16* __restrict__ dout,
                                                    const float* __restrict__ lse, float* __restrict__ ws,
                                                    int B, int H, int S, int Sp) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(B) * H * Sp) return;
  const int s = static_cast<int>(idx % Sp);
  const int bh = static_cast<int>(idx / Sp);
  float d = 0.f, l2 = 0.f;
  if (s < S) {
    const int b = bh / H, h = bh % H;
    const size_t row = ((static_cast<size_t>(b) * S + s) * H + h) * D;
    const uint4* po = reinterpret_cast<const uint4*>(o + row);
    const uint4* pd = reinterpret_cast<const uint4*>(dout + row);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const uint4 a = po[c], g = pd[c];
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        d = fmaf(__uint_as_float(aw[q] << 16), __uint_as_float(gw[q] << 16), d);
        d = fmaf(__uint_as_float(aw[q] & 0xFFFF0000u), __uint_as_float(gw[q] & 0xFFFF0000u), d);
      }
    }
    l2 = lse[static_cast<size_t>(bh) * S + s] * LOG2E;
  }
  ws[static_cast<size_t>(2 * bh) * Sp + s] = d;
  ws[static_cast<size_t>(2 * bh + 1) * Sp + s] = l2;
}

// Shared layout of the two MMA kernels: two resident tiles, a ring of NSTAGE stages (two
// streamed tiles + the 128 rows' Delta and lse*log2e), barriers, TMEM slot, abort flag.
struct BwdSmem {
  uint32_t res0, res1;       // resident tiles
  uint32_t ring;             // stage s at ring + s * STAGE_BYTES
  uint32_t bar0;
  uint8_t* base;
  uint32_t base_u32;
};

// ------------------------------------------------------------ kernel 2: dK and dV --
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int NSTAGE = C::NSTAGE;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const uint32_t sK = base_u32, sV = base_u32 + C::TILE_BYTES;
  const uint32_t ring = base_u32 + 2 * C::TILE_BYTES;
  const uint32_t bar0 = ring + NSTAGE * C::STAGE_BYTES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + (bar0 - base_u32) + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto sQ = [&](int s) { return ring + s * C::STAGE_BYTES; };
  auto sDO = [&](int s) { return ring + s * C::STAGE_BYTES + C::TILE_BYTES; };
  auto vec = [&](int s) {
    return reinterpret_cast<const float*>(base + (ring - base_u32) + s * C::STAGE_BYTES + 2 * C::TILE_BYTES);
  };
  const uint32_t BAR_KV = bar0, BAR_S = bar0 + 8, BAR_P = bar0 + 16, BAR_ACC = bar0 + 24;
  auto BAR_FULL = [&](int s) { return bar0 + 32 + 8u * s; };
  auto BAR_EMPTY = [&](int s) { return bar0 + 32 + 8u * (NSTAGE + s); };
  const uint32_t BAR_DONE = bar0 + 32 + 8u * (2 * NSTAGE);
  // dP^T ready (its own commit, after S^T's), and dS^T written (after P^T's hand-off)
  const uint32_t BAR_DP = BAR_DONE + 8, BAR_DS = BAR_DONE + 16;

  const uint32_t warp = warp_id(), lane = lane_id();
  // CTA -> (key tile, b, key/value head): key tile slowest, so the causal key tiles with the
  // most query tiles start first.  The query heads of the group (G = H / Hkv, head hkv * G + g)
  // all read these keys: iteration i takes query tile j0 + i % nqt of head g = i / nqt, and
  // dK, dV accumulate over all of them.
  const int BH = p.B * p.Hkv, G = p.H / p.Hkv;
  const int kt = static_cast<int>(blockIdx.x) / BH, bkv = static_cast<int>(blockIdx.x) % BH;
  const int b = bkv / p.Hkv, hkv = bkv % p.Hkv;
  const int k0 = 128 * kt;
  const int nq = (p.S + 127) / 128;
  const int j0 = CAUSAL ? kt : 0;          // first query tile that sees these keys
  const int nqt = nq - j0;
  const int ntile = G * nqt;
  auto q_tile = [&](int i) { return j0 + i % nqt; };
  auto q_head = [&](int i) { return hkv * G + i / nqt; };

  // The dQ kernel reads nothing this kernel writes: it may start on SMs this grid leaves
  // idle once every CTA of this grid is running (programmatic dependent launch).
  if (threadIdx.x == 0) grid_launch_dependents();
  if (threadIdx.x == 0) {
    mbar_init(BAR_KV, 1);
    mbar_init(BAR_S, 1);
    mbar_init(BAR_P, C::COMPUTE_WARPS);
    mbar_init(BAR_ACC, 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(BAR_FULL(s), 1);
      mbar_init(BAR_EMPTY(s), 1);
    }
    mbar_init(BAR_DONE, 1);
    mbar_init(BAR_DP, 1);
    mbar_init(BAR_DS, C::COMPUTE_WARPS);
    *abort_flag = 0;
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
      const uint64_t pol_res = l2_policy_evict_first(), pol_str = l2_policy_evict_last();
      mbar_arrive_expect_tx(BAR_KV, 2 * C::TILE_BYTES);
      for (int pn = 0; pn < C::NPANEL; ++pn) {
        tma_load_4d(sK + pn * C::PANEL_BYTES, &tmK, BAR_KV, pn * C::PANEL_ELEMS, hkv, k0, b, pol_res);
        tma_load_4d(sV + pn * C::PANEL_BYTES, &tmV, BAR_KV, pn * C::PANEL_ELEMS, hkv, k0, b, pol_res);
      }
      int i = 0;
      for (; i < ntile && !*abort_flag; ++i) {
        const int s = i % NSTAGE;
        if (!wait_bounded(BAR_EMPTY(s), ((i / NSTAGE) & 1) ^ 1u, ctl, WHERE_BWD_LOAD)) break;
        const int q0 = 128 * q_tile(i), h = q_head(i), bh = b * p.H + h;
        mbar_arrive_expect_tx(BAR_FULL(s), 2 * C::TILE_BYTES + C::VEC_BYTES);
        for (int pn = 0; pn < C::NPANEL; ++pn) {
          tma_load_4d(sQ(s) + pn * C::PANEL_BYTES, &tmQ, BAR_FULL(s), pn * C::PANEL_ELEMS, h, q0, b, pol_str);
          tma_load_4d(sDO(s) + pn * C::PANEL_BYTES, &tmDO, BAR_FULL(s), pn * C::PANEL_ELEMS, h, q0, b, pol_str);
        }
        const uint32_t dv = sDO(s) + C::TILE_BYTES;
        bulk_load(dv, p.ws + static_cast<size_t>(2 * bh) * p.Sp + q0, 512, BAR_FULL(s), pol_str);
        bulk_load(dv + 512, p.ws + static_cast<size_t>(2 * bh + 1) * p.Sp + q0, 512, BAR_FULL(s), pol_str);
      }
      if (*abort_flag) {
        wait_drain(BAR_KV, 0, p.spin_limit);
        for (int t = (i > NSTAGE ? i - NSTAGE : 0); t < i; ++t)
          wait_drain(BAR_FULL(t % NSTAGE), (t / NSTAGE) & 1, p.spin_limit);
      }
    }
  } else if (warp == C::MMA_WARP) {
    if (lane == 0) {
      const uint64_t dK = smem_desc(sK, 16, C::SBO, C::LAYOUT), dV = smem_desc(sV, 16, C::SBO, C::LAYOUT);
      bool ok = wait_bounded(BAR_KV, 0, ctl, WHERE_BWD_MMA);
      for (int i = 0; ok && i < ntile; ++i) {
        const int s = i % NSTAGE;
        ok = wait_bounded(BAR_FULL(s), (i / NSTAGE) & 1, ctl, WHERE_BWD_MMA);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dQk = smem_desc(sQ(s), 16, C::SBO, C::LAYOUT);
        const uint64_t dDOk = smem_desc(sDO(s), 16, C::SBO, C::LAYOUT);
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS_SS; ++kk) {      // S^T = K Q^T
          const uint32_t off = ((kk / C::STEPS_PER_PANEL) * C::PANEL_BYTES + (kk % C::STEPS_PER_PANEL) * 32) >> 4;
          mma_f16_ss(tmem, dK + off, dQk + off, C::IDESC_SS, kk > 0);
        }
        mma_commit(BAR_S);                                // the exponentials start on S^T ...
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS_SS; ++kk) {      // ... while dP^T = V dO^T forms
          const uint32_t off = ((kk / C::STEPS_PER_PANEL) * C::PANEL_BYTES + (kk % C::STEPS_PER_PANEL) * 32) >> 4;
          mma_f16_ss(tmem + 128, dV + off, dDOk + off, C::IDESC_SS, kk > 0);
        }
        mma_commit(BAR_DP);
        const uint64_t dDOn = smem_desc(sDO(s), C::PANEL_BYTES, C::SBO, C::LAYOUT);
        const uint64_t dQn = smem_desc(sQ(s), C::PANEL_BYTES, C::SBO, C::LAYOUT);
        // P^T / dS^T of queries 16kk .. 16kk + 15 sit at 8kk + 32 (kk / 4) (the second half of
        // the queries was written by the second half of the compute warps, over its own S^T)
        ok = wait_bounded(BAR_P, i & 1, ctl, WHERE_BWD_MMA);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS_TS; ++kk) {      // dV += P^T dO, while dS^T forms
          const uint32_t off = (kk * 16 * C::PANEL_ROW) >> 4;
          mma_f16_ts(tmem + 256, tmem + 8u * kk + 32u * (kk / 4), dDOn + off, C::IDESC_TS,
                     (i > 0 || kk > 0) ? 1u : 0u);
        }
        ok = wait_bounded(BAR_DS, i & 1, ctl, WHERE_BWD_MMA);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS_TS; ++kk) {      // dK += dS^T Q
          const uint32_t off = (kk * 16 * C::PANEL_ROW) >> 4;
          mma_f16_ts(tmem + 256 + D, tmem + 128 + 8u * kk + 32u * (kk / 4), dQn + off, C::IDESC_TS,
                     (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(BAR_EMPTY(s));
      }
      if (ok) mma_commit(BAR_ACC);
      mma_commit(BAR_DONE);
      wait_drain(BAR_DONE, 0, p.spin_limit);
    }
  } else {
    // compute warps: thread = key row k0 + r of lane quarter wq, query columns 64 hc .. 64 hc + 63
    const int wq = static_cast<int>(warp) % 4, hc = static_cast<int>(warp) / 4;
    const int r = wq * 32 + static_cast<int>(lane);
    const uint32_t tl = tmem + ((static_cast<uint32_t>(wq) * 32u) << 16);
    const int key = k0 + r;
    bool ok = true;
    for (int i = 0; ok && i < ntile; ++i) {
      const int s = i % NSTAGE;
      const int q0 = 128 * q_tile(i);
      const float* dlt = vec(s);
      const float* l2 = dlt + 128;
      // the stage's Delta / lse came by TMA: acquire them from the stage's own barrier (its
      // phase cannot move on before this warp's P arrival releases the stage)
      if (!warp_wait(BAR_FULL(s), (i / NSTAGE) & 1, ctl, WHERE_BWD_COMPUTE)) { ok = false; break; }
      if (!warp_wait(BAR_S, i & 1, ctl, WHERE_BWD_COMPUTE)) { ok = false; break; }
      tc_fence_after();
      // masks are needed only on the diagonal tile (causal) and the ragged last query tile
      const bool masked = (CAUSAL && q_tile(i) == kt) || q0 + 128 > p.S;
      // P^T of this warp's 64 queries (kept for dS^T), stored as bf16 over its own half of S^T
      // (already read): queries 32c .. 32c + 31 at columns 16c + 32hc, so the two halves'
      // stores never touch each other's S.  dV's MMAs start on them while dP^T is used below.
      float pkeep[2][32];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * hc + cc;
        uint32_t sv[32];
        tmem_ld32(tl + 32u * c, sv);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          // the columns' lse*log2e, four at a time (broadcast reads)
          const float4 l4 = *reinterpret_cast<const float4*>(l2 + 32 * c + e);
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            reg_fence(sv[e + u]);
            float x = fmaf(__uint_as_float(sv[e + u]), p.c_log2, -lv[u]);
            if (masked) {
              const int q = q0 + 32 * c + e + u;
              if (!(q < p.S && (!CAUSAL || key <= q))) x = -INFINITY;
            }
            pkeep[cc][e + u] = ex2(x);
          }
          pk[e / 2] = pack_bf16x2(pkeep[cc][e], pkeep[cc][e + 1]);
          pk[e / 2 + 1] = pack_bf16x2(pkeep[cc][e + 2], pkeep[cc][e + 3]);
        }
        tmem_st16(tl + static_cast<uint32_t>(16 * c + 32 * hc), pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR_P);
      // dS^T = P^T * (dP^T - Delta) over this warp's own half of dP^T, the same way
      if (!warp_wait(BAR_DP, i & 1, ctl, WHERE_BWD_COMPUTE)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * hc + cc;
        uint32_t pv[32];
        tmem_ld32(tl + 128u + 32u * c, pv);
        tmem_wait_ld();
        uint32_t dk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 d4 = *reinterpret_cast<const float4*>(dlt + 32 * c + e);
          const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
          float dd[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            reg_fence(pv[e + u]);
            dd[u] = pkeep[cc][e + u] * (__uint_as_float(pv[e + u]) - dv4[u]);
          }
          dk[e / 2] = pack_bf16x2(dd[0], dd[1]);
          dk[e / 2 + 1] = pack_bf16x2(dd[2], dd[3]);
        }
        tmem_st16(tl + 128u + static_cast<uint32_t>(16 * c + 32 * hc), dk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR_DS);
    }
    if (ok && warp_wait(BAR_ACC, 0, ctl, WHERE_BWD_COMPUTE)) {
      tc_fence_after();
      const bool valid = key < p.S;
      const size_t row = ((static_cast<size_t>(b) * p.S + (valid ? key : 0)) * p.Hkv + hkv) * D;
      {
        const int part = hc;                           // dV (first half of the warps), dK (times the softmax scale)
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(part ? p.dk : p.dv) + row;
        const float mul = part ? p.scale : 1.f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t a[32];
          tmem_ld32(tl + 256u + static_cast<uint32_t>(part * D) + 32u * c, a);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            reg_fence(a[2 * e]);
            reg_fence(a[2 * e + 1]);
            pk[e] = pack_bf16x2(__uint_as_float(a[2 * e]) * mul, __uint_as_float(a[2 * e + 1]) * mul);
          }
          if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) d4[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          }
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

// ------------------------------------------------------------------ kernel 3: dQ --
// CTA = 128 queries of one (b, h).  Q and dO stay in shared memory; K_j and V_j stream through
// rings of their own (K is read by S_j and later by dQ += dS_j K_j, V only by dP_j, so V's slots
// free early).  S is double-buffered in Tensor Memory (the columns beside dQ are free), so the
// MMA warp issues S(j+1) and dP(j+1) while the compute warps still work on tile j, and
// dQ += dS(j) K_j after their dS(j): the compute warps go from tile to tile without waiting
// for the tensor core.  dS(j) is written over S(j)'s own buffer.
template <int D>
struct DqCfg {
  using C = BwdCfg<D>;
  static constexpr int NK = D == 64 ? 4 : 3;             // K slots
  static constexpr int NV = D == 64 ? 4 : 2;             // V slots
  // Q/dO ready, dP ready, dP read, accumulate done, drain; then S ready and dS written per
  // S buffer; then full/empty per K slot and per V slot
  static constexpr int NBAR = 5 + 4 + 2 * NK + 2 * NV;
  static constexpr int SMEM_BYTES = 1024 + (2 + NK + NV) * C::TILE_BYTES + NBAR * 8 + 16;
  static constexpr uint32_t S1 = 384;                    // second S buffer's first column
  static_assert(256 + D <= S1 && S1 + 128 <= 512, "Tensor Memory: S, dP, dQ, second S");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const BwdParams p) {
  using C = BwdCfg<D>;
  using Q = DqCfg<D>;
  constexpr int NK = Q::NK, NV = Q::NV;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const uint32_t sQ = base_u32, sDO = base_u32 + C::TILE_BYTES;
  auto sK = [&](int s) { return base_u32 + (2 + s) * C::TILE_BYTES; };
  auto sV = [&](int s) { return base_u32 + (2 + NK + s) * C::TILE_BYTES; };
  const uint32_t bar0 = base_u32 + (2 + NK + NV) * C::TILE_BYTES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + (bar0 - base_u32) + Q::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t BAR_QD = bar0, BAR_DP = bar0 + 8, BAR_DPR = bar0 + 16, BAR_ACC = bar0 + 24;
  const uint32_t BAR_DONE = bar0 + 32;
  auto BAR_S = [&](int b) { return bar0 + 40 + 8u * b; };          // S(j) of buffer b complete
  auto BAR_DS = [&](int b) { return bar0 + 56 + 8u * b; };         // dS(j) of buffer b written
  auto BAR_KF = [&](int s) { return bar0 + 72 + 8u * s; };
  auto BAR_KE = [&](int s) { return bar0 + 72 + 8u * (NK + s); };
  auto BAR_VF = [&](int s) { return bar0 + 72 + 8u * (2 * NK + s); };
  auto BAR_VE = [&](int s) { return bar0 + 72 + 8u * (2 * NK + NV + s); };
  auto s_col = [&](int j) { return (j & 1) ? Q::S1 : 0u; };        // tile j's S buffer

  const uint32_t warp = warp_id(), lane = lane_id();
  // CTA -> (query tile, b, h): causal query tiles with the most key tiles start first
  const int BH = p.B * p.H;
  const int nq = (p.S + 127) / 128;
  const int qt = CAUSAL ? nq - 1 - static_cast<int>(blockIdx.x) / BH : static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int b = bh / p.H, h = bh % p.H;
  const int hkv = h / (p.H / p.Hkv);       // the key/value head this query head reads
  const int q0 = 128 * qt;
  const int ntile = CAUSAL ? qt + 1 : nq;

  if (threadIdx.x == 0) {
    mbar_init(BAR_QD, 1);
    mbar_init(BAR_DP, 1);
    mbar_init(BAR_DPR, C::COMPUTE_WARPS);
    mbar_init(BAR_ACC, 1);
    mbar_init(BAR_DONE, 1);
    for (int bb = 0; bb < 2; ++bb) {
      mbar_init(BAR_S(bb), 1);
      mbar_init(BAR_DS(bb), C::COMPUTE_WARPS);
    }
    for (int s = 0; s < NK; ++s) {
      mbar_init(BAR_KF(s), 1);
      mbar_init(BAR_KE(s), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(BAR_VF(s), 1);
      mbar_init(BAR_VE(s), 1);
    }
    *abort_flag = 0;
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
      const uint64_t pol_res = l2_policy_evict_first(), pol_str = l2_policy_evict_last();
      mbar_arrive_expect_tx(BAR_QD, 2 * C::TILE_BYTES);
      for (int pn = 0; pn < C::NPANEL; ++pn) {
        tma_load_4d(sQ + pn * C::PANEL_BYTES, &tmQ, BAR_QD, pn * C::PANEL_ELEMS, h, q0, b, pol_res);
        tma_load_4d(sDO + pn * C::PANEL_BYTES, &tmDO, BAR_QD, pn * C::PANEL_ELEMS, h, q0, b, pol_res);
      }
      int nk = 0, nv = 0;                                 // K and V tiles issued
      for (int i = 0; i < ntile && !*abort_flag; ++i) {
        const int ks = i % NK, vs = i % NV;
        if (!wait_bounded(BAR_KE(ks), ((i / NK) & 1) ^ 1u, ctl, WHERE_BWD_LOAD)) break;
        mbar_arrive_expect_tx(BAR_KF(ks), C::TILE_BYTES);
        for (int pn = 0; pn < C::NPANEL; ++pn)
          tma_load_4d(sK(ks) + pn * C::PANEL_BYTES, &tmK, BAR_KF(ks), pn * C::PANEL_ELEMS, hkv, 128 * i, b, pol_str);
        ++nk;
        if (!wait_bounded(BAR_VE(vs), ((i / NV) & 1) ^ 1u, ctl, WHERE_BWD_LOAD)) break;
        mbar_arrive_expect_tx(BAR_VF(vs), C::TILE_BYTES);
        for (int pn = 0; pn < C::NPANEL; ++pn)
          tma_load_4d(sV(vs) + pn * C::PANEL_BYTES, &tmV, BAR_VF(vs), pn * C::PANEL_ELEMS, hkv, 128 * i, b, pol_str);
        ++nv;
      }
      if (*abort_flag) {
        // copies still in flight land before the CTA exits
        wait_drain(BAR_QD, 0, p.spin_limit);
        for (int t = (nk > NK ? nk - NK : 0); t < nk; ++t) wait_drain(BAR_KF(t % NK), (t / NK) & 1, p.spin_limit);
        for (int t = (nv > NV ? nv - NV : 0); t < nv; ++t) wait_drain(BAR_VF(t % NV), (t / NV) & 1, p.spin_limit);
      }
    }
  } else if (warp == C::MMA_WARP) {
    if (lane == 0) {
      const uint64_t dQ = smem_desc(sQ, 16, C::SBO, C::LAYOUT), dDO = smem_desc(sDO, 16, C::SBO, C::LAYOUT);
      auto issue_s = [&](int j) -> bool {                // S(j) = Q K_j^T into its buffer
        if (!wait_bounded(BAR_KF(j % NK), (j / NK) & 1, ctl, WHERE_BWD_MMA)) return false;
        tc_fence_after();
        const uint64_t dKk = smem_desc(sK(j % NK), 16, C::SBO, C::LAYOUT);
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS_SS; ++kk) {
          const uint32_t off = ((kk / C::STEPS_PER_PANEL) * C::PANEL_BYTES + (kk % C::STEPS_PER_PANEL) * 32) >> 4;
          mma_f16_ss(tmem + s_col(j), dQ + off, dKk + off, C::IDESC_SS, kk > 0);
        }
        mma_commit(BAR_S(j & 1));
        return true;
      };
      auto issue_dp = [&](int j) -> bool {               // dP(j) = dO V_j^T; V_j's slot then frees
        if (!wait_bounded(BAR_VF(j % NV), (j / NV) & 1, ctl, WHERE_BWD_MMA)) return false;
        tc_fence_after();
        const uint64_t dVk = smem_desc(sV(j % NV), 16, C::SBO, C::LAYOUT);
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS_SS; ++kk) {
          const uint32_t off = ((kk / C::STEPS_PER_PANEL) * C::PANEL_BYTES + (kk % C::STEPS_PER_PANEL) * 32) >> 4;
          mma_f16_ss(tmem + 128, dDO + off, dVk + off, C::IDESC_SS, kk > 0);
        }
        mma_commit(BAR_DP);
        mma_commit(BAR_VE(j % NV));
        return true;
      };
      bool ok = wait_bounded(BAR_QD, 0, ctl, WHERE_BWD_MMA) && issue_s(0) && issue_dp(0);
      for (int i = 0; ok && i < ntile; ++i) {
        if (i + 1 < ntile) {
          // S(i+1) into the other buffer: its last dS (tile i-1) was read by dQ(i-1), issued
          // before; dP(i+1) over dP(i) once the compute warps have read dP(i)
          if (!issue_s(i + 1)) { ok = false; break; }
          if (!wait_bounded(BAR_DPR, i & 1, ctl, WHERE_BWD_MMA)) { ok = false; break; }
          if (!issue_dp(i + 1)) { ok = false; break; }
        }
        if (!wait_bounded(BAR_DS(i & 1), (i >> 1) & 1, ctl, WHERE_BWD_MMA)) { ok = false; break; }
        tc_fence_after();
        const uint64_t dKn = smem_desc(sK(i % NK), C::PANEL_BYTES, C::SBO, C::LAYOUT);
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS_TS; ++kk) {      // dQ += dS K
          const uint32_t off = (kk * 16 * C::PANEL_ROW) >> 4;
          // dS of keys 16kk .. 16kk + 15 at 8kk + 32 (kk / 4) of tile i's buffer
          mma_f16_ts(tmem + 256, tmem + s_col(i) + 8u * kk + 32u * (kk / 4), dKn + off, C::IDESC_TS,
                     (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(BAR_KE(i % NK));
      }
      if (ok) mma_commit(BAR_ACC);
      mma_commit(BAR_DONE);
      wait_drain(BAR_DONE, 0, p.spin_limit);
    }
  } else {
    // compute warps: thread = query row q0 + r of lane quarter wq, key columns 64 hc .. 64 hc + 63
    const int wq = static_cast<int>(warp) % 4, hc = static_cast<int>(warp) / 4;
    const int r = wq * 32 + static_cast<int>(lane);
    const uint32_t tl = tmem + ((static_cast<uint32_t>(wq) * 32u) << 16);
    const int qrow = q0 + r;
    const bool valid = qrow < p.S;
    const float dlt = valid ? p.ws[static_cast<size_t>(2 * bh) * p.Sp + qrow] : 0.f;
    const float l2 = valid ? p.ws[static_cast<size_t>(2 * bh + 1) * p.Sp + qrow] : 0.f;
    bool ok = true;
    for (int i = 0; ok && i < ntile; ++i) {
      const int kb = 128 * i;
      const bool masked = (CAUSAL && i == qt) || kb + 128 > p.S;
      const uint32_t ts = tl + s_col(i);
      if (!warp_wait(BAR_S(i & 1), (i >> 1) & 1, ctl, WHERE_BWD_COMPUTE)) { ok = false; break; }
      tc_fence_after();
      // P of this warp's 64 keys, while the tensor core may still be forming dP
      float pkeep[2][32];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * hc + cc;
        uint32_t sv[32];
        tmem_ld32(ts + 32u * c, sv);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          reg_fence(sv[e]);
          float x = fmaf(__uint_as_float(sv[e]), p.c_log2, -l2);
          if (masked) {
            const int kcol = kb + 32 * c + e;
            if (!(kcol < p.S && (!CAUSAL || kcol <= qrow))) x = -INFINITY;
          }
          pkeep[cc][e] = ex2(x);
        }
      }
      if (!warp_wait(BAR_DP, i & 1, ctl, WHERE_BWD_COMPUTE)) { ok = false; break; }
      tc_fence_after();
      uint32_t pv[2][32];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) tmem_ld32(tl + 128u + 32u * (2 * hc + cc), pv[cc]);
      tmem_wait_ld();
      // dP(i) is in registers: the MMA warp may form dP(i+1) over it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR_DPR);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * hc + cc;
        uint32_t dk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          reg_fence(pv[cc][e]);
          reg_fence(pv[cc][e + 1]);
          dk[e / 2] = pack_bf16x2(pkeep[cc][e] * (__uint_as_float(pv[cc][e]) - dlt),
                                  pkeep[cc][e + 1] * (__uint_as_float(pv[cc][e + 1]) - dlt));
        }
        // dS over this warp's own half of S (already read): keys 32c .. 32c + 31 at 16c + 32hc
        tmem_st16(ts + static_cast<uint32_t>(16 * c + 32 * hc), dk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR_DS(i & 1));
    }
    if (ok && warp_wait(BAR_ACC, 0, ctl, WHERE_BWD_COMPUTE)) {
      tc_fence_after();
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.dq) +
                           ((static_cast<size_t>(b) * p.S + (valid ? qrow : 0)) * p.H + h) * D;
#pragma unroll 1
      for (int c = hc * (D / 64); c < (hc + 1) * (D / 64); ++c) {   // this warp's half of dQ's columns
        uint32_t a[32];
        tmem_ld32(tl + 256u + 32u * c, a);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          reg_fence(a[2 * e]);
          reg_fence(a[2 * e + 1]);
          pk[e] = pack_bf16x2(__uint_as_float(a[2 * e]) * p.scale, __uint_as_float(a[2 * e + 1]) * p.scale);
        }
        if (valid) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) d4[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
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
  // This grid may have started before the dK/dV grid finished (programmatic dependent launch);
  // it ends only after that grid has completed and its writes are visible, so the stream's
  // next operation sees every gradient.
  grid_dependency_wait();
}

template <int D, bool CAUSAL>
cudaError_t launch_bwd_d(const CUtensorMap* maps, const BwdParams& p, cudaStream_t st) {
  using C = BwdCfg<D>;
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if ((configured.load() & bit) == 0) {
    e = cudaFuncSetAttribute(bwd_dkdv_kernel<D, CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(bwd_dq_kernel<D, CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               DqCfg<D>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  const long long rows = static_cast<long long>(p.B) * p.H * p.Sp;
  delta_kernel<D><<<static_cast<unsigned>((rows + 255) / 256), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(p.o), static_cast<const __nv_bfloat16*>(p.dout), p.lse, p.ws, p.B, p.H,
      p.S, p.Sp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const unsigned nqt = static_cast<unsigned>((p.S + 127) / 128);
  // dK/dV: one CTA per (key tile, b, key/value head); dQ: one per (query tile, b, query head)
  bwd_dkdv_kernel<D, CAUSAL><<<static_cast<unsigned>(p.B * p.Hkv) * nqt, C::THREADS, C::SMEM_BYTES, st>>>(
      maps[0], maps[1], maps[2], maps[3], p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // dQ after dK/dV with programmatic stream serialization: its CTAs take the SMs the last,
  // partly filled wave of dK/dV CTAs leaves idle (the two kernels never share an SM: each
  // needs most of its shared memory)
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B * p.H) * nqt);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = DqCfg<D>::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, bwd_dq_kernel<D, CAUSAL>, maps[0], maps[1], maps[2], maps[3], p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd(const CUtensorMap* maps, const BwdParams& p, int D, bool causal, cudaStream_t st) {
  if (D == 64) return causal ? launch_bwd_d<64, true>(maps, p, st) : launch_bwd_d<64, false>(maps, p, st);
  return causal ? launch_bwd_d<128, true>(maps, p, st) : launch_bwd_d<128, false>(maps, p, st);
}

}  // namespace ea46
