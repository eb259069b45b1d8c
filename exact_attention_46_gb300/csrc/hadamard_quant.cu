// hadamard_quant.cu -- random-sign Hadamard rotation + per-block E4M3 quantisation.
//
// What it computes ("FlashAttention-3 (NL)", "Technische innovaties", item 3; hada.io FA3
// summary, "Niedrige FP8-Präzision und incoherent processing"): every D-element row x of a
// [B, S, H, D] bf16 tensor becomes x' = (x * signs) H_D / sqrt(D) (H_D the Sylvester
// Hadamard matrix; no rotation when signs is null), each (b, h, 128-token block) gets one
// scale = amax(|x'|) / 448 (1 for an all-zero block), and out = E4M3(x' / scale), rounded to
// nearest even and saturating.
//
// Design: the transform is O(D log D) per row and the kernel is bound by HBM traffic
// (2 bytes read + 1 byte written per element), so it stays on the FP32 pipes: no tensor
// cores.  One CTA = one (b, h, token block) = 128 rows; 4 lanes share a row, each holding
// D/4 elements chosen so that every 16-byte load of a row segment is contiguous across the
// 4 lanes (element index = 32*i + 8*part + e).  Butterflies over index bits 0-2 (e) and
// 5.. (i) stay inside a thread; bits 3-4 (part) take two shuffle stages.  The block amax is
// a warp shuffle reduction plus one shared-memory pass; values stay in registers between
// the two phases, so the input is read exactly once.
#include <cstdint>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ea46 {

namespace {

constexpr int QROWS = 128;            // tokens per scale block
constexpr int QTHREADS = QROWS * 4;   // 4 lanes per row

template <int D, bool ROTATE>
__global__ void __launch_bounds__(QTHREADS)
    hadamard_quant_kernel(const QuantParams p) {
  constexpr int NI = D / 32;          // 16-byte groups per thread
  constexpr int VPT = D / 4;          // values per thread
  __shared__ float warp_max[QTHREADS / 32];

  const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int part = lane & 3;
  const int r = warp * 8 + (lane >> 2);          // row within the block
  const int tok = blk * QROWS + r;
  const bool valid = tok < p.S;
  const size_t row_off = (static_cast<size_t>(b) * p.S + (valid ? tok : 0)) * p.H + h;

  float v[VPT];
  const uint4* src = reinterpret_cast<const uint4*>(
      reinterpret_cast<const __nv_bfloat16*>(p.x) + row_off * D);
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    uint4 w = valid ? __ldg(src + 4 * i + part) : make_uint4(0, 0, 0, 0);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[8 * i + 2 * k] = __uint_as_float(ws[k] << 16);
      v[8 * i + 2 * k + 1] = __uint_as_float(ws[k] & 0xFFFF0000u);
    }
  }

  if (ROTATE) {
    const float4* sg = reinterpret_cast<const float4*>(p.signs);
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const float4 s0 = __ldg(sg + 8 * i + 2 * part);
      const float4 s1 = __ldg(sg + 8 * i + 2 * part + 1);
      v[8 * i + 0] *= s0.x; v[8 * i + 1] *= s0.y; v[8 * i + 2] *= s0.z; v[8 * i + 3] *= s0.w;
      v[8 * i + 4] *= s1.x; v[8 * i + 5] *= s1.y; v[8 * i + 6] *= s1.z; v[8 * i + 7] *= s1.w;
    }
    // index bits 0-2: inside each 8-group
#pragma unroll
    for (int hs = 1; hs < 8; hs <<= 1)
#pragma unroll
      for (int i = 0; i < NI; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if ((e & hs) == 0) {
            const float a = v[8 * i + e], c = v[8 * i + e + hs];
            v[8 * i + e] = a + c;
            v[8 * i + e + hs] = a - c;
          }
    // index bits 3-4: across the 4 lanes of the row
#pragma unroll
    for (int lm = 1; lm < 4; lm <<= 1) {
      const bool upper = (part & lm) != 0;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const float o = __shfl_xor_sync(0xffffffffu, v[k], lm);
        v[k] = upper ? (o - v[k]) : (v[k] + o);
      }
    }
    // index bits 5..: across the 8-groups of a thread
#pragma unroll
    for (int is = 1; is < NI; is <<= 1)
#pragma unroll
      for (int i = 0; i < NI; ++i)
        if ((i & is) == 0)
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float a = v[8 * i + e], c = v[8 * i + is * 8 + e];
            v[8 * i + e] = a + c;
            v[8 * i + is * 8 + e] = a - c;
          }
  }

  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < VPT; ++k) amax = fmaxf(amax, fabsf(v[k]));
  if (!valid) amax = 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) warp_max[warp] = amax;
  __syncthreads();
  amax = warp_max[0];
#pragma unroll
  for (int w = 1; w < QTHREADS / 32; ++w) amax = fmaxf(amax, warp_max[w]);

  // x' = y / sqrt(D); scale = amax(x') / 448; code = E4M3(x' / scale) = E4M3(y * 448 / amax(y)).
  const float inv = amax > 0.f ? 448.f / amax : 0.f;
  if (threadIdx.x == 0) {
    const float norm = ROTATE ? rsqrtf(static_cast<float>(D)) : 1.f;
    p.scale[(static_cast<size_t>(b) * p.H + h) * p.nblk + blk] =
        amax > 0.f ? (amax * norm) / 448.f : 1.f;
  }
  if (valid) {
    uint2* dst = reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(p.out) + row_off * D);
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const uint32_t lo = pack_e4m3x4(v[8 * i] * inv, v[8 * i + 1] * inv, v[8 * i + 2] * inv,
                                      v[8 * i + 3] * inv);
      const uint32_t hi = pack_e4m3x4(v[8 * i + 4] * inv, v[8 * i + 5] * inv,
                                      v[8 * i + 6] * inv, v[8 * i + 7] * inv);
      dst[4 * i + part] = make_uint2(lo, hi);
    }
  }
}

}  // namespace

template <int D>
cudaError_t launch_hadamard_quant(const QuantParams& p, cudaStream_t stream) {
  const dim3 grid(p.nblk, p.H, p.B);
  if (p.signs != nullptr)
    hadamard_quant_kernel<D, true><<<grid, QTHREADS, 0, stream>>>(p);
  else
    hadamard_quant_kernel<D, false><<<grid, QTHREADS, 0, stream>>>(p);
  return cudaGetLastError();
}

template cudaError_t launch_hadamard_quant<64>(const QuantParams&, cudaStream_t);
template cudaError_t launch_hadamard_quant<128>(const QuantParams&, cudaStream_t);
template cudaError_t launch_hadamard_quant<256>(const QuantParams&, cudaStream_t);

}  // namespace ea46
