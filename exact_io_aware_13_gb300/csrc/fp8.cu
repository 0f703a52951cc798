// Quantisation of bf16 attention inputs to e4m3 with block scales, for the FP8
// forward ("FlashAttention/es", "Variantes y sucesores", names FP8 for FlashAttention-3;
// "FlashAttention-3 y torch.compile", section 2, its block quantisation).
//
// Q and K: one fp32 scale per 128-row tile of a head, s = amax / 448 (1 if the tile is
// all zero), code = e4m3(x / s) with an IEEE fp32 division and round-to-nearest-even
// (448 is the largest finite e4m3 value, so nothing saturates but a rounding overshoot).
// V: one scale per head, and the codes are written transposed, [d, keys] with the key
// count padded to a multiple of 16 (padding is zero), because the P V product reads V
// K-major. The reductions are maxima, so every result is independent of the launch.
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kRowsPerTile = 128;
constexpr int kThreadsQ = 256;
constexpr float kE4m3Max = 448.0f;

__device__ __forceinline__ float bf16_abs_max8(uint4 w) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
  float m = 0.f;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float2 f = __bfloat1622float2(h[t]);
    m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
  }
  return m;
}

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
    red[32] = m;
  }
  __syncthreads();
  return red[32];
}

// Eight bf16 values / s to eight e4m3 codes (two 32-bit words, lowest element first).
__device__ __forceinline__ uint2 quant8(uint4 w, float s) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
  uint32_t r[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const float2 a = __bfloat1622float2(h[2 * q]), b = __bfloat1622float2(h[2 * q + 1]);
    r[q] = pack_e4m3x2(a.x / s, a.y / s) | (pack_e4m3x2(b.x / s, b.y / s) << 16);
  }
  return make_uint2(r[0], r[1]);
}

// One CTA per (head, 128-row tile).
__global__ void __launch_bounds__(kThreadsQ) quant_tiles_kernel(const __nv_bfloat16* x,
                                                                 uint8_t* out, float* scales,
                                                                 int N, int d, int ntiles) {
  __shared__ float red[33];
  const int tile = blockIdx.x, bh = blockIdx.y;
  const int r0 = tile * kRowsPerTile, rows = imin(kRowsPerTile, N - r0);
  const int per_row = d / 8;  // 16-byte chunks per row
  const size_t base = ((size_t)bh * N + r0) * d;
  const uint4* src = reinterpret_cast<const uint4*>(x + base);
  float m = 0.f;
  for (int c = threadIdx.x; c < rows * per_row; c += kThreadsQ) m = fmaxf(m, bf16_abs_max8(src[c]));
  const float amax = block_max(m, red);
  const float s = amax > 0.f ? amax / kE4m3Max : 1.f;
  uint2* dst = reinterpret_cast<uint2*>(out + base);
  for (int c = threadIdx.x; c < rows * per_row; c += kThreadsQ) dst[c] = quant8(src[c], s);
  if (threadIdx.x == 0) scales[(size_t)bh * ntiles + tile] = s;
}

// One CTA per head: the head's amax, then 128-key blocks transposed through shared
// memory into [d, npad] rows of e4m3 codes.
__global__ void __launch_bounds__(kThreadsQ) quant_v_kernel(const __nv_bfloat16* x,
                                                             uint8_t* out, float* scales,
                                                             int N, int d, int npad) {
  __shared__ float red[33];
  __shared__ __align__(16) __nv_bfloat16 blk[kRowsPerTile][128 + 8];  // [key][dim], padded rows
  const int bh = blockIdx.x;
  const int per_row = d / 8;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)bh * N * d);
  float m = 0.f;
  for (size_t c = threadIdx.x; c < (size_t)N * per_row; c += kThreadsQ)
    m = fmaxf(m, bf16_abs_max8(src[c]));
  const float amax = block_max(m, red);
  const float s = amax > 0.f ? amax / kE4m3Max : 1.f;
  uint8_t* dhead = out + (size_t)bh * d * npad;
  for (int j0 = 0; j0 < npad; j0 += kRowsPerTile) {
    __syncthreads();
    for (int c = threadIdx.x; c < kRowsPerTile * per_row; c += kThreadsQ) {
      const int jj = c / per_row, cc = c % per_row, j = j0 + jj;
      const uint4 w = j < N ? src[(size_t)j * per_row + cc] : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(&blk[jj][cc * 8]) = w;
    }
    __syncthreads();
    // output row `dim`, keys j0 + 16 q .. + 15 (16 codes per thread and step)
    const int keys = imin(kRowsPerTile, npad - j0);
    for (int c = threadIdx.x; c < d * (keys / 16); c += kThreadsQ) {
      const int dim = c / (keys / 16), q = c % (keys / 16);
      uint32_t wv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int jj = q * 16 + 4 * e;
        const float f0 = __bfloat162float(blk[jj][dim]), f1 = __bfloat162float(blk[jj + 1][dim]);
        const float f2 = __bfloat162float(blk[jj + 2][dim]), f3 = __bfloat162float(blk[jj + 3][dim]);
        wv[e] = pack_e4m3x2(f0 / s, f1 / s) | (pack_e4m3x2(f2 / s, f3 / s) << 16);
      }
      *reinterpret_cast<uint4*>(dhead + (size_t)dim * npad + j0 + q * 16) =
          make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
  }
  if (threadIdx.x == 0) scales[bh] = s;
}

}  // namespace

cudaError_t launch_quantize_tiles(const __nv_bfloat16* x, uint8_t* out, float* scales, int BH,
                                  int N, int d, cudaStream_t st) {
  if (BH == 0 || N == 0) return cudaSuccess;
  const int ntiles = ceil_div(N, kRowsPerTile);
  if (BH > 65535) return cudaErrorInvalidValue;
  quant_tiles_kernel<<<dim3(ntiles, BH), kThreadsQ, 0, st>>>(x, out, scales, N, d, ntiles);
  return cudaGetLastError();
}

cudaError_t launch_quantize_v_transposed(const __nv_bfloat16* x, uint8_t* out, float* scales,
                                         int BH, int N, int d, cudaStream_t st) {
  if (BH == 0) return cudaSuccess;
  const int npad = (N + 15) / 16 * 16;
  quant_v_kernel<<<BH, kThreadsQ, 0, st>>>(x, out, scales, N, d, npad);
  return cudaGetLastError();
}

}  // namespace attn
