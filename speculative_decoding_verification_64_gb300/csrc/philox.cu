// Uniforms on the device: the Philox4x64-10 counter-based generator
// (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
// SC'11), for the u_i ~ U(0,1) of the accept tests and the final draw
// ("Chapter 15: Decoding acceleration", section 15.1.2 step 3).
//
// One round maps the counter block (x0, x1, x2, x3) with key (k0, k1) to
//     (hi(M1 x2) ^ x1 ^ k0,  lo(M1 x2),  hi(M0 x0) ^ x3 ^ k1,  lo(M0 x0)),
// hi/lo being the halves of the 128-bit product; the key is bumped by the
// Weyl constants between rounds; ten rounds.  Word i of the stream that starts
// from counter c is word i mod 4 of the block for counter c + floor(i/4) + 1
// (256-bit, little-endian 64-bit words; the counter advances before each
// block, as NumPy's Philox bit generator does), and u_i = ((w_i >> 41) + 0.5)
// * 2^-23, exact in float32 and strictly inside (0, 1).  One thread makes one
// block of four words.
#include "common.cuh"

namespace specdec {
namespace {

constexpr uint64_t kM0 = 0xD2E7470EE14C6C93ull;
constexpr uint64_t kM1 = 0xCA5A826395121157ull;
constexpr uint64_t kW0 = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kW1 = 0xBB67AE8584CAA73Bull;
constexpr int kThreads = 256;

__device__ __forceinline__ void philox_block(uint64_t x[4], uint64_t k0, uint64_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += kW0;
      k1 += kW1;
    }
    const uint64_t lo0 = kM0 * x[0], hi0 = __umul64hi(kM0, x[0]);
    const uint64_t lo1 = kM1 * x[2], hi1 = __umul64hi(kM1, x[2]);
    const uint64_t y0 = hi1 ^ x[1] ^ k0, y2 = hi0 ^ x[3] ^ k1;
    x[0] = y0;
    x[1] = lo1;
    x[2] = y2;
    x[3] = lo0;
  }
}

// x += a (256-bit)
__device__ __forceinline__ void add256(uint64_t x[4], uint64_t a) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint64_t v = x[i] + a;
    a = (v < x[i]) ? 1ull : 0ull;
    x[i] = v;
  }
}

__global__ void __launch_bounds__(kThreads) philox_uniforms_kernel(const PhiloxParams p) {
  const uint64_t j = p.first / 4 + (uint64_t)blockIdx.x * kThreads + threadIdx.x;  // block
  const uint64_t last = p.first + (uint64_t)(p.n - 1);  // last word (no overflow: host check)
  if (j > last / 4) return;
  uint64_t x[4] = {p.counter[0], p.counter[1], p.counter[2], p.counter[3]};
  add256(x, j);
  add256(x, 1);
  philox_block(x, p.key[0], p.key[1]);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint64_t w = j * 4 + t;
    if (w >= p.first && w <= last)
      p.out[w - p.first] = ((float)(uint32_t)(x[t] >> 41) + 0.5f) * 0x1p-23f;
  }
}

}  // namespace

cudaError_t launch_philox_uniforms(const PhiloxParams &p, cudaStream_t stream) {
  if (p.n <= 0) return cudaSuccess;
  const uint64_t b0 = p.first / 4, b1 = (p.first + (uint64_t)(p.n - 1)) / 4;
  const uint64_t blocks = b1 - b0 + 1;
  const uint64_t grid = (blocks + kThreads - 1) / kThreads;
  philox_uniforms_kernel<<<(unsigned)grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace specdec
