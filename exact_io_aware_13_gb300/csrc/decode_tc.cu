// Decode entry point (no row copies and the launcher), and the kernel that merges the
// partial results of the key chunks and row copies by their log-sum-exp.
#include "decode_tc.cuh"

namespace attn {
namespace dec {

// One warp per output row: merge the partial results of the chunks that hold keys of
// the row, in chunk order.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const Args a) {
  const DecodeProblem& p = a.p;
  const long long grow = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (grow >= a.rows_total) return;
  const int b = (int)(grow / ((long long)p.Hq * p.Nq));
  const int i = (int)(grow % p.Nq);
  int Lb = p.seq_lens[b];
  Lb = Lb < 0 ? 0 : (Lb > p.max_seq_len ? p.max_seq_len : Lb);
  int lo, hi;
  decode_row_keys(p.mask_kind, p.window, Lb, p.Nq, i, lo, hi);
  constexpr int kPer = D / 32;  // columns per lane
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  float M = -INFINITY, W = 0.f;
  if (hi > lo) {
    const int ca = lo / p.chunk, cb = (hi - 1) / p.chunk + 1;
    const int pa = ca * a.rep, pb = cb * a.rep;  // partial results of chunks [ca, cb)
    for (int cc = pa + lane; cc < pb; cc += 32)
      M = fmaxf(M, a.out.part_lse[(size_t)cc * a.rows_total + grow]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (M > -INFINITY) {
      for (int cc = pa; cc < pb; ++cc) {
        const float w = ex2_approx(a.out.part_lse[(size_t)cc * a.rows_total + grow] - M);
        W += w;
        const float* src = a.out.part_o + ((size_t)cc * a.rows_total + grow) * D + lane * kPer;
        if constexpr (kPer == 4) {
          const float4 v = *reinterpret_cast<const float4*>(src);
          acc[0] = fmaf(w, v.x, acc[0]);
          acc[1] = fmaf(w, v.y, acc[1]);
          acc[2] = fmaf(w, v.z, acc[2]);
          acc[3] = fmaf(w, v.w, acc[3]);
        } else {
          const float2 v = *reinterpret_cast<const float2*>(src);
          acc[0] = fmaf(w, v.x, acc[0]);
          acc[1] = fmaf(w, v.y, acc[1]);
        }
      }
    }
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  __nv_bfloat16* dst = a.out.o + grow * D + lane * kPer;
  if constexpr (kPer == 4) {
    uint2 w;
    w.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    w.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = w;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
  if (lane == 0) a.out.lse[grow] = W > 0.f ? (M + log2f(W)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace dec

cudaError_t launch_decode_tc(const DecodeProblem& p, const CUtensorMap& tk, const CUtensorMap& tv,
                             const DecodeOut& out, int num_ctas, cudaStream_t st) {
  using namespace dec;
  Args a{};
  a.p = p;
  a.out = out;
  a.G = p.Hq / p.Hkv;
  a.rows = a.G * p.Nq;
  a.row_tiles = ceil_div(a.rows, kItemRows);
  a.rep = decode_row_copies(a.rows);
  a.n_part = (a.rep == 2 || a.rows > 32) ? 2 : 1;
  a.rows_total = (long long)p.B * p.Hq * p.Nq;
  a.direct = p.n_chunks == 1 && a.rep == 1;
  if (a.rows_total == 0 || num_ctas <= 0) return cudaSuccess;
  if ((a.rows_total + 7) / 8 > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaError_t e = a.rep == 2 ? launch_decode_copies2(a, tk, tv, num_ctas, st)
                             : launch_decode_copies<1>(a, tk, tv, num_ctas, st);
  if (e != cudaSuccess || a.direct) return e;
  const long long blocks = (a.rows_total + 7) / 8;
  if (p.d == 64) decode_combine_kernel<64><<<(unsigned)blocks, 256, 0, st>>>(a);
  else decode_combine_kernel<128><<<(unsigned)blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace attn
