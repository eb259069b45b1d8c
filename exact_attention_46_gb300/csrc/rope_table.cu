// rope_table.cu -- the rotary-embedding table read by the fused RoPE + rotation + quantiser.
//
// RoPE as in RoFormer (Su et al. 2021, section 3.2), the reading taken for the rotary embedding
// that the hada.io FA3 summary ("Niedrige FP8-Präzision und incoherent processing") names as
// the bandwidth-bound op to fuse the Hadamard rotation with: pair i of the row at position p
// turns by p * theta_i, theta_i = base^(-2i/D).  Entry (p, i) of the table is
// (cos, sin)(p * theta_i), evaluated in fp64 and rounded to nearest fp32, so that every entry
// is the fp32 value closest to the exact one (up to the fp64 library's last-bit error).  The
// table is built once per (n_pos, D, base) and reused across calls; its cost is not on the
// per-step path.
#include <cuda_runtime.h>

#include "internal.h"

namespace ea46 {

namespace {

__global__ void rope_table_kernel(float2* cs, long long n, int D, double base) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= n) return;
  const long long p = idx / (D / 2);
  const int i = static_cast<int>(idx % (D / 2));
  const double theta = pow(base, -2.0 * i / D);
  double s, c;
  sincos(static_cast<double>(p) * theta, &s, &c);
  cs[idx] = make_float2(__double2float_rn(c), __double2float_rn(s));
}

}  // namespace

cudaError_t launch_rope_table(float* cs, int n_pos, int D, double base, cudaStream_t stream) {
  const long long n = static_cast<long long>(n_pos) * (D / 2);
  const int threads = 256;
  const long long blocks = (n + threads - 1) / threads;
  rope_table_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      reinterpret_cast<float2*>(cs), n, D, base);
  return cudaGetLastError();
}

}  // namespace ea46
