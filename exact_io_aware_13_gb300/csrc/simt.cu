// CUDA-core kernels: a one-thread-per-row forward and backward used to cross-check
// the tensor-core kernels, the backward's row term D, and the tile classifier.
//
// The forward follows the online-softmax recurrence of "FlashAttention/es"
// ("El truco del softmax en línea"): a running max m and normaliser l per row, the
// partial output rescaled by exp(m_old - m_new) whenever the max grows. Here the
// recurrence advances one key at a time, in fp32 with accurate expf/tanhf.
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kRows = 128;   // query rows (or keys) per block
constexpr int kKeys = 32;    // keys staged in shared memory per step

struct ScoreOut { float s; float dcap; };  // modified score; d(capped)/d(pre-cap)

__device__ __forceinline__ ScoreOut simt_score(float dot, int i, int j, const Problem& p,
                                               float slope) {
  float s = dot * p.scale;
  if (p.score_kind & ATTN_SCORE_ALIBI) s -= slope * (float)(i - j);
  float dcap = 1.0f;
  if (p.score_kind & ATTN_SCORE_SOFTCAP) {
    const float t = tanhf(s / p.softcap);
    s = p.softcap * t;
    dcap = 1.0f - t * t;
  }
  return {s, dcap};
}

template <int D>
__global__ void __launch_bounds__(kRows) fwd_simt_kernel(Problem p, const __nv_bfloat16* q,
                                                         const __nv_bfloat16* k,
                                                         const __nv_bfloat16* v,
                                                         __nv_bfloat16* o, float* lse) {
  __shared__ float ks[kKeys][D];
  __shared__ float vs[kKeys][D];
  const int bh = blockIdx.y, b = bh / p.Hq, h = bh % p.Hq, g = h / (p.Hq / p.Hkv);
  const int r0 = blockIdx.x * kRows;
  const int i = r0 + threadIdx.x;
  const bool row_ok = i < p.Nq;
  const __nv_bfloat16* qrow = q + ((size_t)bh * p.Nq + (row_ok ? i : 0)) * D;
  const __nv_bfloat16* kh = k + (size_t)(b * p.Hkv + g) * p.Nkv * D;
  const __nv_bfloat16* vh = v + (size_t)(b * p.Hkv + g) * p.Nkv * D;
  float qf[D], acc[D];
#pragma unroll
  for (int c = 0; c < D; ++c) { qf[c] = __bfloat162float(qrow[c]); acc[c] = 0.f; }
  const float slope = alibi_slope(h, p.Hq);
  const int fk = row_ok ? first_key(p.mask, i) : 0;
  float m = -INFINITY, l = 0.f;
  const TileRange tr = kv_tiles_for_rows(p.mask, r0, kRows);
  const int kbeg = tr.lo * kRows, kend = imin(tr.hi * kRows, p.Nkv);
  for (int j0 = kbeg; j0 < kend; j0 += kKeys) {
    __syncthreads();
    for (int e = threadIdx.x; e < kKeys * D; e += kRows) {
      const int jj = e / D, c = e % D, j = j0 + jj;
      ks[jj][c] = j < p.Nkv ? __bfloat162float(kh[(size_t)j * D + c]) : 0.f;
      vs[jj][c] = j < p.Nkv ? __bfloat162float(vh[(size_t)j * D + c]) : 0.f;
    }
    __syncthreads();
    if (!row_ok) continue;
    for (int jj = 0; jj < kKeys; ++jj) {
      const int j = j0 + jj;
      if (!allowed(p.mask, i, j, fk)) continue;
      float dot = 0.f;
#pragma unroll
      for (int c = 0; c < D; ++c) dot = fmaf(qf[c], ks[jj][c], dot);
      const float s = simt_score(dot, i, j, p, slope).s;
      const float m_new = fmaxf(m, s);
      const float corr = expf(m - m_new);  // 0 when m = -inf
      const float e = expf(s - m_new);
      l = l * corr + e;
#pragma unroll
      for (int c = 0; c < D; ++c) acc[c] = acc[c] * corr + e * vs[jj][c];
      m = m_new;
    }
  }
  if (!row_ok) return;
  __nv_bfloat16* orow = o + ((size_t)bh * p.Nq + i) * D;
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int c = 0; c < D; ++c) orow[c] = __float2bfloat16_rn(acc[c] * inv);
  lse[(size_t)bh * p.Nq + i] = l > 0.f ? m + logf(l) : -INFINITY;
}

// dQ: one thread per query row, over the keys the row may see.
template <int D>
__global__ void __launch_bounds__(kRows) dq_simt_kernel(Problem p, const __nv_bfloat16* q,
                                                        const __nv_bfloat16* k,
                                                        const __nv_bfloat16* v,
                                                        const float* lse,
                                                        const __nv_bfloat16* dout,
                                                        const float* delta,
                                                        __nv_bfloat16* dq) {
  __shared__ float ks[kKeys][D];
  __shared__ float vs[kKeys][D];
  const int bh = blockIdx.y, b = bh / p.Hq, h = bh % p.Hq, g = h / (p.Hq / p.Hkv);
  const int r0 = blockIdx.x * kRows;
  const int i = r0 + threadIdx.x;
  const bool row_ok = i < p.Nq;
  const size_t row = (size_t)bh * p.Nq + (row_ok ? i : 0);
  const __nv_bfloat16* kh = k + (size_t)(b * p.Hkv + g) * p.Nkv * D;
  const __nv_bfloat16* vh = v + (size_t)(b * p.Hkv + g) * p.Nkv * D;
  float qf[D], dof[D], acc[D];
#pragma unroll
  for (int c = 0; c < D; ++c) {
    qf[c] = __bfloat162float(q[row * D + c]);
    dof[c] = __bfloat162float(dout[row * D + c]);
    acc[c] = 0.f;
  }
  const float L = lse[row], Di = delta[(size_t)bh * p.nq_pad + (row_ok ? i : 0)];
  const float slope = alibi_slope(h, p.Hq);
  const int fk = row_ok ? first_key(p.mask, i) : 0;
  const TileRange tr = kv_tiles_for_rows(p.mask, r0, kRows);
  const int kbeg = tr.lo * kRows, kend = imin(tr.hi * kRows, p.Nkv);
  for (int j0 = kbeg; j0 < kend; j0 += kKeys) {
    __syncthreads();
    for (int e = threadIdx.x; e < kKeys * D; e += kRows) {
      const int jj = e / D, c = e % D, j = j0 + jj;
      ks[jj][c] = j < p.Nkv ? __bfloat162float(kh[(size_t)j * D + c]) : 0.f;
      vs[jj][c] = j < p.Nkv ? __bfloat162float(vh[(size_t)j * D + c]) : 0.f;
    }
    __syncthreads();
    if (!row_ok || L == -INFINITY) continue;
    for (int jj = 0; jj < kKeys; ++jj) {
      const int j = j0 + jj;
      if (!allowed(p.mask, i, j, fk)) continue;
      float dot = 0.f, dp = 0.f;
#pragma unroll
      for (int c = 0; c < D; ++c) {
        dot = fmaf(qf[c], ks[jj][c], dot);
        dp = fmaf(dof[c], vs[jj][c], dp);
      }
      const ScoreOut so = simt_score(dot, i, j, p, slope);
      const float pr = expf(so.s - L);
      const float ds = pr * (dp - Di) * so.dcap;
#pragma unroll
      for (int c = 0; c < D; ++c) acc[c] = fmaf(ds, ks[jj][c], acc[c]);
    }
  }
  if (!row_ok) return;
#pragma unroll
  for (int c = 0; c < D; ++c) dq[row * D + c] = __float2bfloat16_rn(acc[c] * p.scale);
}

// dK, dV: one thread per key, over the query heads of its group and the rows that
// may see the key.
template <int D>
__global__ void __launch_bounds__(kRows) dkdv_simt_kernel(Problem p, const __nv_bfloat16* q,
                                                          const __nv_bfloat16* k,
                                                          const __nv_bfloat16* v,
                                                          const float* lse,
                                                          const __nv_bfloat16* dout,
                                                          const float* delta,
                                                          __nv_bfloat16* dk,
                                                          __nv_bfloat16* dv) {
  __shared__ float qs[kKeys][D];
  __shared__ float ds_[kKeys][D];
  __shared__ float ls[kKeys], dls[kKeys];
  const int bg = blockIdx.y, b = bg / p.Hkv, g = bg % p.Hkv, G = p.Hq / p.Hkv;
  const int k0 = blockIdx.x * kRows;
  const int j = k0 + threadIdx.x;
  const bool key_ok = j < p.Nkv;
  const size_t krow = (size_t)bg * p.Nkv + (key_ok ? j : 0);
  float kf[D], vf[D], dka[D], dva[D];
#pragma unroll
  for (int c = 0; c < D; ++c) {
    kf[c] = __bfloat162float(k[krow * D + c]);
    vf[c] = __bfloat162float(v[krow * D + c]);
    dka[c] = 0.f; dva[c] = 0.f;
  }
  const TileRange tr = q_tiles_for_keys(p.mask, k0, kRows);
  const int rbeg = tr.lo * kRows, rend = imin(tr.hi * kRows, p.Nq);
  for (int h = g * G; h < (g + 1) * G; ++h) {
    const size_t qh = (size_t)(b * p.Hq + h) * p.Nq;
    const float slope = alibi_slope(h, p.Hq);
    for (int i0 = rbeg; i0 < rend; i0 += kKeys) {
      __syncthreads();
      for (int e = threadIdx.x; e < kKeys * D; e += kRows) {
        const int ii = e / D, c = e % D, i = i0 + ii;
        qs[ii][c] = i < p.Nq ? __bfloat162float(q[(qh + i) * D + c]) : 0.f;
        ds_[ii][c] = i < p.Nq ? __bfloat162float(dout[(qh + i) * D + c]) : 0.f;
      }
      if (threadIdx.x < kKeys) {
        const int i = i0 + threadIdx.x;
        ls[threadIdx.x] = i < p.Nq ? lse[qh + i] : -INFINITY;
        dls[threadIdx.x] = i < p.Nq ? delta[(size_t)(b * p.Hq + h) * p.nq_pad + i] : 0.f;
      }
      __syncthreads();
      if (!key_ok) continue;
      for (int ii = 0; ii < kKeys; ++ii) {
        const int i = i0 + ii;
        if (i >= p.Nq || ls[ii] == -INFINITY) continue;
        if (!allowed(p.mask, i, j, first_key(p.mask, i))) continue;
        float dot = 0.f, dp = 0.f;
#pragma unroll
        for (int c = 0; c < D; ++c) {
          dot = fmaf(qs[ii][c], kf[c], dot);
          dp = fmaf(ds_[ii][c], vf[c], dp);
        }
        const ScoreOut so = simt_score(dot, i, j, p, slope);
        const float pr = expf(so.s - ls[ii]);
        const float dsv = pr * (dp - dls[ii]) * so.dcap;
#pragma unroll
        for (int c = 0; c < D; ++c) {
          dva[c] = fmaf(pr, ds_[ii][c], dva[c]);
          dka[c] = fmaf(dsv, qs[ii][c], dka[c]);
        }
      }
    }
  }
  if (!key_ok) return;
#pragma unroll
  for (int c = 0; c < D; ++c) {
    dk[krow * D + c] = __float2bfloat16_rn(dka[c] * p.scale);
    dv[krow * D + c] = __float2bfloat16_rn(dva[c]);
  }
}

// Row terms of the backward (see RowTerms). A block takes kBlockRows padded query rows of
// one head (16 KB of O and 16 KB of dO rows: nq_pad is a multiple of 128, so a block never
// straddles two heads), copies the valid rows of O and dO into shared memory with two bulk
// copies (so a few blocks per SM keep a few hundred KB in flight), and then one group of
// D/8 lanes per row multiplies its 16-byte pieces and sums them with a fixed butterfly, so
// D_i does not depend on the launch.
template <int D>
struct RowdotShape {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kBlockRows = 16384 / kRowBytes;  // 128, 64 or 32 rows
  static constexpr int kThreads = 128;
  static constexpr int kLanes = D / 8;                   // lanes per row
  static constexpr int kGroups = 32 / kLanes;            // rows per warp and pass
  static constexpr int kPasses = kBlockRows / (kThreads / 32) / kGroups;
};

template <int D>
__global__ void __launch_bounds__(128) rowdot_kernel(Problem p, const __nv_bfloat16* o,
                                                     const __nv_bfloat16* dout,
                                                     const float* lse, RowTerms rt) {
  using S = RowdotShape<D>;
  __shared__ alignas(128) uint8_t rows_o[S::kBlockRows * S::kRowBytes];
  __shared__ alignas(128) uint8_t rows_do[S::kBlockRows * S::kRowBytes];
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  const int blocks_per_head = p.nq_pad / S::kBlockRows;
  const long long bh = blockIdx.x / blocks_per_head;
  const int i0 = (int)(blockIdx.x - bh * blocks_per_head) * S::kBlockRows;
  const int nvalid = imax(0, imin(S::kBlockRows, p.Nq - i0));
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && nvalid > 0) {
    const uint32_t bytes = (uint32_t)nvalid * S::kRowBytes;
    const size_t src = ((size_t)bh * p.Nq + i0) * D;
    mbar_arrive_expect_tx(smem_u32(&bar), 2 * bytes);
    bulk_load(smem_u32(rows_o), o + src, bytes, smem_u32(&bar));
    bulk_load(smem_u32(rows_do), dout + src, bytes, smem_u32(&bar));
  }
  const WaitCtx wc{&abort_flag, p.status};
  const bool have = nvalid == 0 || mbar_wait(smem_u32(&bar), 0, wc);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = lane / S::kLanes, sub = lane % S::kLanes;
#pragma unroll
  for (int ps = 0; ps < S::kPasses; ++ps) {
    const int r = (warp * S::kPasses + ps) * S::kGroups + grp;  // row in the block
    const int i = i0 + r;
    const bool real = r < nvalid;
    float s = 0.f;
    if (real && have) {
      const uint4 av = reinterpret_cast<const uint4*>(rows_o + r * S::kRowBytes)[sub];
      const uint4 bv = reinterpret_cast<const uint4*>(rows_do + r * S::kRowBytes)[sub];
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&av);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&bv);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 x = __bfloat1622float2(a2[t]), y = __bfloat1622float2(b2[t]);
        s = fmaf(x.x, y.x, s);
        s = fmaf(x.y, y.y, s);
      }
    }
#pragma unroll
    for (int off = S::kLanes / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (sub == 0) {
      const long long row = bh * p.nq_pad + i;
      float l2 = INFINITY;
      if (real) {
        const float L = lse[(size_t)bh * p.Nq + i];
        l2 = L == -INFINITY ? INFINITY : L * 1.4426950408889634f;
      }
      rt.delta[row] = real ? s * p.drop_keep : 0.f;  // with dropout D (1 - p)
      rt.lse2[row] = l2;
      if (bh == 0) rt.first[i] = real ? first_key(p.mask, i) : 0x7fffffff;
    }
  }
  // No copy may land in shared memory after the block has left.
  if (threadIdx.x == 0 && nvalid > 0 && !have) drain_wait(smem_u32(&bar), 0);
}

// Rows with no key at all: O = 0, lse = -inf.
__global__ void fill_masked_kernel(long long rows, int d, __nv_bfloat16* o, float* lse) {
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < rows * d;
       t += (long long)gridDim.x * blockDim.x) {
    o[t] = __float2bfloat16_rn(0.f);
    if (t % d == 0) lse[t / d] = -INFINITY;
  }
}

__global__ void classify_kernel(MaskSpec m, int32_t* classes) {
  const int nkt = ceil_div(m.nkv, ATTN_TILE), nqt = ceil_div(m.nq, ATTN_TILE);
  const long long total = (long long)nqt * nkt;
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (long long)gridDim.x * blockDim.x) {
    const int qt = (int)(t / nkt), kt = (int)(t % nkt);
    classes[t] = tile_class(m, qt, kt, ATTN_TILE);
  }
}

}  // namespace

cudaError_t launch_fwd_simt(const Problem& p, const __nv_bfloat16* q, const __nv_bfloat16* k,
                            const __nv_bfloat16* v, __nv_bfloat16* o, float* lse,
                            cudaStream_t st) {
  dim3 grid(ceil_div(p.Nq, kRows), p.B * p.Hq);
  if (p.d == 64) fwd_simt_kernel<64><<<grid, kRows, 0, st>>>(p, q, k, v, o, lse);
  else fwd_simt_kernel<128><<<grid, kRows, 0, st>>>(p, q, k, v, o, lse);
  return cudaGetLastError();
}

cudaError_t launch_bwd_simt(const Problem& p, const __nv_bfloat16* q, const __nv_bfloat16* k,
                            const __nv_bfloat16* v, const float* lse, const __nv_bfloat16* dout,
                            const float* delta, __nv_bfloat16* dq, __nv_bfloat16* dk,
                            __nv_bfloat16* dv, cudaStream_t st) {
  if (p.Nq > 0) {
    dim3 g1(ceil_div(p.Nq, kRows), p.B * p.Hq);
    if (p.d == 64) dq_simt_kernel<64><<<g1, kRows, 0, st>>>(p, q, k, v, lse, dout, delta, dq);
    else dq_simt_kernel<128><<<g1, kRows, 0, st>>>(p, q, k, v, lse, dout, delta, dq);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.Nkv == 0) return e;
  dim3 g2(ceil_div(p.Nkv, kRows), p.B * p.Hkv);
  if (p.d == 64)
    dkdv_simt_kernel<64><<<g2, kRows, 0, st>>>(p, q, k, v, lse, dout, delta, dk, dv);
  else
    dkdv_simt_kernel<128><<<g2, kRows, 0, st>>>(p, q, k, v, lse, dout, delta, dk, dv);
  return cudaGetLastError();
}

cudaError_t launch_bwd_rowdot(const Problem& p, const __nv_bfloat16* o,
                              const __nv_bfloat16* dout, const float* lse, const RowTerms& rt,
                              cudaStream_t st) {
  const long long rows = (long long)p.B * p.Hq * p.nq_pad;
  if (rows == 0) return cudaSuccess;
  const int block_rows = 16384 / (p.d * 2);  // RowdotShape<d>::kBlockRows
  const long long blocks = rows / block_rows;  // nq_pad is a multiple of 128
  if (blocks > 0x7fffffffLL || p.nq_pad % block_rows != 0) return cudaErrorInvalidValue;
  if (p.d == 64) rowdot_kernel<64><<<(unsigned)blocks, 128, 0, st>>>(p, o, dout, lse, rt);
  else if (p.d == 128) rowdot_kernel<128><<<(unsigned)blocks, 128, 0, st>>>(p, o, dout, lse, rt);
  else rowdot_kernel<256><<<(unsigned)blocks, 128, 0, st>>>(p, o, dout, lse, rt);
  return cudaGetLastError();
}

cudaError_t launch_fill_masked(long long rows, int d, __nv_bfloat16* o, float* lse,
                               cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  fill_masked_kernel<<<1024, 256, 0, st>>>(rows, d, o, lse);
  return cudaGetLastError();
}

cudaError_t launch_classify(const MaskSpec& m, int32_t* classes, cudaStream_t st) {
  const long long total = (long long)ceil_div(m.nq, ATTN_TILE) * ceil_div(m.nkv, ATTN_TILE);
  if (total == 0) return cudaSuccess;
  const int blocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
  classify_kernel<<<blocks, 256, 0, st>>>(m, classes);
  return cudaGetLastError();
}

}  // namespace attn
