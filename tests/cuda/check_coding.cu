// Exhaustive GPU self-test of the quantizers' E4M3 coding of x / S.
//
// For every BF16 amax (all 32768 non-negative bit patterns that are finite)
// the scale S is formed as the kernels form it, and every finite BF16 x with
// |x| <= amax (the values a group with that amax can hold) is coded with the
// kernels' coding routines -- both the binary32 form and the BF16-word form;
// each result must equal the code of the correctly rounded binary32 division
// RN32(x / S) (CUDA's __fdiv_rn).  This covers the whole input domain of the
// weight, activation and amax-recalibrating KV quantizers.  Prints the
// mismatch count and the first mismatch.
#include <cstdint>
#include <cstdio>

#include "../../w8a8_gemm_rl_gb300/csrc/common.cuh"

using namespace w8a8;

__global__ void check(unsigned long long* bad, unsigned int* first) {
  const uint32_t a_bits = blockIdx.x;  // 0 .. 0x7FFF: non-negative BF16 patterns
  const float amax = __uint_as_float(a_bits << 16);
  if (!isfinite(amax)) return;
  const float S = scale_from_amax(amax);
  const QuantScale qs = make_quant_scale(S);
  unsigned long long local = 0;
  for (uint32_t base = threadIdx.x * 4; base < 65536; base += blockDim.x * 4) {
    float x[4];
    uint32_t xb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      xb[i] = base + i;
      x[i] = __uint_as_float(xb[i] << 16);
      if (!isfinite(x[i]) || fabsf(x[i]) > amax) {  // outside the domain: use 0
        xb[i] = 0;
        x[i] = 0.0f;
      }
    }
    const uint32_t c = quant_f32x4(x[0], x[1], x[2], x[3], qs);
    const uint32_t cw = quant_bf16x4(xb[0] | (xb[1] << 16), xb[2] | (xb[3] << 16), qs);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t want = code_exact(x[i], S);
      if (((c >> (8 * i)) & 0xFFu) != want || ((cw >> (8 * i)) & 0xFFu) != want) {
        ++local;
        atomicCAS(first, 0xFFFFFFFFu, (a_bits << 16) | (base + i));
      }
    }
  }
  if (local) atomicAdd(bad, local);
}

int main() {
  unsigned long long* bad;
  unsigned int* first;
  if (cudaMalloc(&bad, sizeof(*bad)) != cudaSuccess || cudaMalloc(&first, sizeof(*first)) != cudaSuccess)
    return 2;
  cudaMemset(bad, 0, sizeof(*bad));
  cudaMemset(first, 0xFF, sizeof(*first));
  check<<<32768, 256>>>(bad, first);
  cudaError_t e = cudaDeviceSynchronize();
  unsigned long long hb = 0;
  unsigned int hf = 0;
  cudaMemcpy(&hb, bad, sizeof(hb), cudaMemcpyDeviceToHost);
  cudaMemcpy(&hf, first, sizeof(hf), cudaMemcpyDeviceToHost);
  printf("status %s mismatches %llu first_amax_bits 0x%04x first_x_bits 0x%04x\n", cudaGetErrorString(e),
         hb, hf >> 16, hf & 0xFFFFu);
  return (e == cudaSuccess && hb == 0) ? 0 : 1;
}
