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
//     S = Q K_j^T and O += P V_j on the tensor core; four warps (thread = tile row) run the
//     online softmax as the prefill kernel does (lazy rescale, P as bf16 over S);
//   * S is double-buffered in Tensor Memory and S(j+1) is issued before PV(j), so the softmax
//     of tile j overlaps the next QK^T and the chain per tile shortens to the slower of the
//     two.  The one hazard -- a lazy rescale of O while PV(j-1) still accumulates -- is closed
//     by a PV-done barrier that the softmax waits on only when it rescales.
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

template <int D>
struct DecCfg {
  static constexpr int ROW_BYTES = D * 2;
  static constexpr int PANEL_ROW = 128;
  static constexpr int NPANEL = ROW_BYTES / PANEL_ROW;
  static constexpr int PANEL_ELEMS = 64;
  static constexpr int PANEL_BYTES = 128 * PANEL_ROW;
  static constexpr int TILE_BYTES = 128 * ROW_BYTES;
  static constexpr int NSLOT = D == 64 ? 12 : 6;               // K/V tiles in flight
  static constexpr uint32_t SBO = 8 * PANEL_ROW;
  static constexpr uint32_t LAYOUT = 2u;
  static constexpr int KSTEPS_QK = ROW_BYTES / 32;
  static constexpr int STEPS_PER_PANEL = PANEL_ROW / 32;
  static constexpr int KSTEPS_PV = 128 / 16;
  static constexpr uint32_t IDESC_QK = instr_desc(1, 0, 128, 128);
  static constexpr uint32_t IDESC_PV = instr_desc(1, 1, 128, D);
  static constexpr int NBAR = 8 + 2 * NSLOT;
  static constexpr int SMEM_BYTES = 1024 + (1 + NSLOT) * TILE_BYTES + NBAR * 8 + 16;
  static constexpr int THREADS = 32 * 6;
  static constexpr int LOAD_WARP = 4, MMA_WARP = 5;
  static_assert(D == 64 || D == 128, "head dimension");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

enum : int { WHERE_DEC_LOAD = 21, WHERE_DEC_MMA = 22, WHERE_DEC_SOFTMAX = 23 };

__device__ __forceinline__ void wait_drain_dec(uint32_t bar, uint32_t parity, long long limit) {
  if (mbar_try_wait(bar, parity)) return;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > limit) return;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(DecCfg<D>::THREADS, 1)
    attn_decode_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
  using C = DecCfg<D>;
  constexpr int NSLOT = C::NSLOT;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const uint32_t sQ = base_u32;
  const uint32_t sKV = base_u32 + C::TILE_BYTES;
  const uint32_t bar0 = sKV + NSLOT * C::TILE_BYTES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + (bar0 - base_u32) + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t BAR_Q = bar0, BAR_O = bar0 + 8, BAR_DONE = bar0 + 16, BAR_PV = bar0 + 24;
  auto BAR_S = [&](int b2) { return bar0 + 32 + 8u * b2; };       // S buffer b2 written
  auto BAR_P = [&](int b2) { return bar0 + 48 + 8u * b2; };       // P in buffer b2 written
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
  const int R = p.G * p.Sq;                  // packed query rows (<= 128)

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
    fence_barrier_init();
  }
  if (warp == C::MMA_WARP) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // S buffers at columns 0 and 128 (P over the first 64 of each), O at 256
  const uint32_t tmem = *tmem_slot;
  constexpr uint32_t O_COL = 256;
  const WaitCtl ctl{p.spin_limit, abort_flag, p.err_word, p.err_info};

  if (warp == C::LOAD_WARP) {
    if (lane == 0) {
      const uint64_t pol_q = l2_policy_evict_first(), pol_kv = l2_policy_evict_first();
      mbar_arrive_expect_tx(BAR_Q, C::NPANEL * R * C::PANEL_ROW);
      for (int pn = 0; pn < C::NPANEL; ++pn)
        tma_load_5d(sQ + pn * C::PANEL_BYTES, &tmQ, BAR_Q, pn * C::PANEL_ELEMS, 0, hkv, 0, b, pol_q);
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
          mma_f16_ss(tmem + 128u * (j & 1), dq + off, bk + off, C::IDESC_QK, kk > 0);
        }
        mma_commit(BAR_S(j & 1));
        mma_commit(BAR_EMPTY(ks));
        return true;
      };
      if (ok) ok = qk(0);
      for (int j = 0; ok && j < ntile; ++j) {
        // S(j+1) goes into the other buffer, whose P(j-1) was read by PV(j-1) (issued earlier)
        if (j + 1 < ntile && !(ok = qk(j + 1))) break;
        if (!(ok = wait_bounded(BAR_P(j & 1), (j >> 1) & 1, ctl, WHERE_DEC_MMA))) break;
        const int idx = 2 * j + 1, vs = idx % NSLOT;
        if (!(ok = wait_bounded(BAR_FULL(vs), (idx / NSLOT) & 1, ctl, WHERE_DEC_MMA))) break;
        tc_fence_after();
        const uint64_t bv = dv0 + ((vs * C::TILE_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS_PV; ++kk) {
          const uint32_t off = (kk * 16 * C::PANEL_ROW) >> 4;
          mma_f16_ts(tmem + O_COL, tmem + 128u * (j & 1) + 8u * kk, bv + off, C::IDESC_PV,
                     (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(BAR_PV);
        mma_commit(BAR_EMPTY(vs));
      }
      if (ok) mma_commit(BAR_O);
      mma_commit(BAR_DONE);
      wait_drain_dec(BAR_DONE, 0, p.spin_limit);
    }
  } else {
    // softmax warps: thread = packed row r = (token r / G, head r % G)
    const int r = static_cast<int>(warp) * 32 + static_cast<int>(lane);
    const uint32_t tl = tmem + ((warp * 32u) << 16);
    const int tok = r / p.G;
    const int lim_all = p.Sk - p.Sq + tok;    // last visible key under the mask
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < ntile; ++j) {
      const int kb = 128 * (t0 + j);
      const uint32_t sb = tl + 128u * (j & 1);
      if (!wait_bounded(BAR_S(j & 1), (j >> 1) & 1, ctl, WHERE_DEC_SOFTMAX)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(sb + 32u * c, sr[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) reg_fence(sr[c][i]);
      // visible keys of this tile: kb + col <= lim (lim < 0: none)
      const int lim = (CAUSAL ? (lim_all < p.Sk - 1 ? lim_all : p.Sk - 1) : p.Sk - 1) - kb;
      if (lim < 127) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * c + i > lim) sr[c][i] = __float_as_uint(-INFINITY);
      }
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; i += 2) mt = max3(mt, __uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1]));
      mt *= p.c_log2;
      bool rescale = false;
      float alpha = 1.f;
      if (mt > m_run + TAU_DEC || (m_run == -INFINITY && mt != -INFINITY)) {
        alpha = m_run == -INFINITY ? 0.f : ex2(m_run - mt);
        m_run = mt;
        l_run *= alpha;
        rescale = j > 0;
      }
      const float off = m_run == -INFINITY ? 0.f : m_run;   // no visible key yet: p = 0
      float ls = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ex2(fmaf(__uint_as_float(sr[c][2 * i]), p.c_log2, -off));
          const float p1 = ex2(fmaf(__uint_as_float(sr[c][2 * i + 1]), p.c_log2, -off));
          ls += p0 + p1;
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16(sb + 16u * c, pk);
      }
      l_run += ls;
      if (__any_sync(0xffffffffu, rescale)) {
        // O must hold PV(j-1) complete (PV(j) waits for this warp's arrival below); S(j) may
        // have been issued before PV(j-1), so wait for PV(j-1)'s completion explicitly
        if (!wait_bounded(BAR_PV, (j - 1) & 1, ctl, WHERE_DEC_SOFTMAX)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tl + O_COL + 32u * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            reg_fence(o[i]);
            o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          }
          tmem_st32(tl + O_COL + 32u * c, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR_P(j & 1));
    }
    if (ok && wait_bounded(BAR_O, 0, ctl, WHERE_DEC_SOFTMAX)) {
      tc_fence_after();
      const bool valid = r < R;
      const int g = r % p.G, h = hkv * p.G + g;
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      const float lse = l_run > 0.f ? (m_run + __log2f(l_run)) * LN2_DEC : -INFINITY;
      const size_t row = (static_cast<size_t>(b) * p.Hq + h) * p.Sq + (valid ? tok : 0);   // [B, Hq, Sq]
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tl + O_COL + 32u * c, o);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) reg_fence(o[i]);
        if (!valid) continue;
        if (p.n_split == 1) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) +
                                                ((static_cast<size_t>(b) * p.Sq + tok) * p.Hq + h) * D + 32 * c);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
        } else {
          float4* dst = reinterpret_cast<float4*>(p.ws_o + (static_cast<size_t>(split) * p.rows_total + row) * D + 32 * c);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            dst[v4] = make_float4(__uint_as_float(o[4 * v4]) * inv_l, __uint_as_float(o[4 * v4 + 1]) * inv_l,
                                  __uint_as_float(o[4 * v4 + 2]) * inv_l, __uint_as_float(o[4 * v4 + 3]) * inv_l);
        }
      }
      if (valid) {
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

template <int D, bool CAUSAL>
cudaError_t launch_decode_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const DecodeParams& p, cudaStream_t st) {
  using C = DecCfg<D>;
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if ((configured.load() & bit) == 0) {
    e = cudaFuncSetAttribute(attn_decode_kernel<D, CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  const unsigned grid = static_cast<unsigned>(p.B * p.Hkv * p.n_split);
  attn_decode_kernel<D, CAUSAL><<<grid, C::THREADS, C::SMEM_BYTES, st>>>(tq, tk, tv, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.n_split > 1) {
    const long long threads = p.rows_total * 32;
    decode_combine_kernel<D><<<static_cast<unsigned>((threads + 255) / 256), 256, 0, st>>>(p);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace

cudaError_t launch_attn_decode(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeParams& p, int D, bool causal, cudaStream_t st) {
  if (D == 64) return causal ? launch_decode_d<64, true>(tq, tk, tv, p, st) : launch_decode_d<64, false>(tq, tk, tv, p, st);
  return causal ? launch_decode_d<128, true>(tq, tk, tv, p, st) : launch_decode_d<128, false>(tq, tk, tv, p, st);
}

}  // namespace ea46
