"""The e4m3 quantisation of h divides by its scale through the correctly rounded reciprocal plus
one correction step (``div_rn_by_recip`` in the library's ``common.cuh``).  It must give the same
fp32 quotient as an IEEE division, so that the quantisation decision stays the one the oracle
takes in fp32.  This test compiles a small probe against the library header, runs it on 2^28
inputs shaped like the quantisation (|x| <= amax, s = amax / 448, amax over 120 binades), and
requires no difference in the quotient or in the e4m3 code."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "mixture_experts_ffn_gemm_gb300", "csrc")

PROBE = r'''
#include <cstdio>
#include <cstdint>
#include "common.cuh"
using namespace moe;

__device__ uint32_t mix(uint32_t a) {
  a ^= a >> 16; a *= 0x7feb352dU; a ^= a >> 15; a *= 0x846ca68bU; a ^= a >> 16; return a;
}
__global__ void probe(uint64_t n, unsigned long long* bad, unsigned long long* bad_code) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += stride) {
    const uint32_t h1 = mix((uint32_t)i * 2u + 1u), h2 = mix(h1 ^ (uint32_t)(i >> 20));
    const float amax = __uint_as_float(((h1 & 0x3fffffffu) % (120u << 23)) + (67u << 23));
    const float frac = __uint_as_float((h2 & 0x007fffffu) | 0x3f000000u);
    const int sh = (h2 >> 23) & 31;
    float x = amax * frac * __uint_as_float((127u - sh) << 23);
    if (h2 >> 31) x = -x;
    if ((h1 >> 30) == 3u) x = (h2 & 1u) ? -amax : amax;
    const float s = __fdiv_rn(amax, 448.0f);
    const float a = __fdiv_rn(x, s), b = div_rn_by_recip(x, s, __frcp_rn(s));
    if (__float_as_uint(a) != __float_as_uint(b)) {
      atomicAdd(bad, 1ull);
      unsigned short qa, qb;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(qa) : "f"(0.f), "f"(a));
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(qb) : "f"(0.f), "f"(b));
      if (qa != qb) atomicAdd(bad_code, 1ull);
    }
  }
}
int main() {
  unsigned long long* d;
  unsigned long long h[2] = {1, 1};
  if (cudaMalloc(&d, 16) != cudaSuccess) return 2;
  cudaMemset(d, 0, 16);
  probe<<<152 * 8, 256>>>(1ull << 28, d, d + 1);
  if (cudaDeviceSynchronize() != cudaSuccess) return 3;
  cudaMemcpy(h, d, 16, cudaMemcpyDeviceToHost);
  printf("%llu %llu\n", h[0], h[1]);
  return 0;
}
'''


@pytest.mark.gpu
def test_reciprocal_division_matches_ieee_division(cuda_device, tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    src = tmp_path / "div_probe.cu"
    src.write_text(PROBE)
    exe = tmp_path / "div_probe"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "--expt-relaxed-constexpr", "-I", CSRC, str(src), "-o", str(exe)],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    quotient_mismatches, code_mismatches = int(out[0]), int(out[1])
    assert quotient_mismatches == 0
    assert code_mismatches == 0
