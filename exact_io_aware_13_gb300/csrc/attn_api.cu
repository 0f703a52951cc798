// The C ABI of libattn.so: argument checks, TMA tensor maps, the device status
// word, and the launch sequence of each entry point. Nothing here allocates device
// memory; every buffer comes from the caller.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "attn.h"
#include "kernels.h"
#include "ptx.cuh"

namespace attn {
namespace {
// Failure-path self-test: thread 0 waits on a fresh mbarrier that nothing arrives on,
// with the same bounded wait as every kernel; it gives up after kWaitLimitNs, raising
// the CTA's abort flag and DEV_TIMEOUT in the library's status word, and returns.
__global__ void selftest_wait_kernel(int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncwarp();
  WaitCtx wc{&abort_flag, status};
  if (threadIdx.x == 0) (void)mbar_wait(smem_u32(&bar), 0, wc);
  __syncwarp();
}


// Check of a document-offsets table, one thread per entry: offs[0] = 0, non-decreasing,
// offs[n_docs] = n. A violation sets DEV_BAD_INPUT in the status word. Reads only
// offs[0 .. n_docs].
__global__ void doc_offsets_check_kernel(const int32_t* offs, int n_docs, int n, int* status) {
  const long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (k > n_docs) return;
  const int v = offs[k];
  const bool bad = (k == 0 && v != 0) || (k == n_docs && v != n) ||
                   (k < n_docs && offs[k + 1] < v);
  if (bad) atomicOr(status, DEV_BAD_INPUT);
}


// Sticky device status word of this library (one per device that loads it).
__device__ int g_device_status;

constexpr int kMaxDevices = 64;
// Bit of the device status word that bounded waits set (DEV_TIMEOUT in the kernels);
// any other set bit reports an out-of-range device input.
constexpr int DEV_TIMEOUT_BIT = 1;

struct DeviceInfo {
  bool probed = false;
  bool is_sm103 = false;
  int* status = nullptr;  // device address of g_device_status on this device
  int num_sms = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Device checks and per-device state, done once per device with it current.
attn_status current_device(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.probed) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return ATTN_ERR_LAUNCH;
    d.is_sm103 = (major == 10 && minor == 3);
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATTN_ERR_LAUNCH;
    if (d.is_sm103) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_device_status) != cudaSuccess) return ATTN_ERR_LAUNCH;
      d.status = static_cast<int*>(ptr);
      if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
          return ATTN_ERR_LAUNCH;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
      }
    }
    d.probed = true;
  }
  if (!d.is_sm103) return ATTN_ERR_ARCH;
  *out = &d;
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Shared argument checks of the forward and backward entry points; fills `p`.
attn_status check_problem(int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale,
                          int mask_kind, const attn_mask_params* mp, int score_kind,
                          const attn_score_params* sp, Problem* p) {
  if (B < 0 || Hq < 0 || Hkv < 0 || Nq < 0 || Nkv < 0) return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_SHAPE;  // 256: tensor-core forward only
  if (Hkv == 0 ? Hq != 0 : (Hq % Hkv) != 0) return ATTN_ERR_SHAPE;
  const long long rows_q = (long long)B * Hq * Nq, rows_k = (long long)B * Hkv * Nkv;
  if (rows_q * d > 0x7fffffffLL * 16 || rows_k * d > 0x7fffffffLL * 16) return ATTN_ERR_SHAPE;
  if ((long long)B * Hq > 0x7fffffff / 2) return ATTN_ERR_SHAPE;
  if (!std::isfinite(scale)) return ATTN_ERR_ARG;
  if (mask_kind < ATTN_MASK_NONE || mask_kind > ATTN_MASK_DOCUMENT_CAUSAL) return ATTN_ERR_ARG;
  if (score_kind & ~(ATTN_SCORE_ALIBI | ATTN_SCORE_SOFTCAP | ATTN_SCORE_DROPOUT))
    return ATTN_ERR_ARG;
  std::memset(p, 0, sizeof(*p));
  p->B = B; p->Hq = Hq; p->Hkv = Hkv; p->Nq = Nq; p->Nkv = Nkv; p->d = d;
  p->scale = scale;
  p->score_kind = score_kind;
  p->mask.kind = mask_kind;
  p->mask.nq = Nq;
  p->mask.nkv = Nkv;
  p->nq_pad = (int)(((long long)Nq + 127) / 128 * 128);
  if (score_kind & ATTN_SCORE_SOFTCAP) {
    if (!sp || !(sp->softcap > 0.f) || !std::isfinite(sp->softcap)) return ATTN_ERR_ARG;
    p->softcap = sp->softcap;
  }
  p->drop_scale = 1.f;
  p->drop_keep = 1.f;
  if (score_kind & ATTN_SCORE_DROPOUT) {
    if (!sp || !(sp->dropout_p >= 0.f && sp->dropout_p < 1.f)) return ATTN_ERR_ARG;
    p->drop_thr = std::min(255, (int)std::floor(sp->dropout_p * 256.0f));
    p->drop_keep = 1.0f - sp->dropout_p;
    p->drop_scale = 1.0f / p->drop_keep;
    p->drop_seed_lo = (uint32_t)(sp->dropout_seed & 0xFFFFFFFFull);
    p->drop_seed_hi = (uint32_t)(sp->dropout_seed >> 32);
  }
  if (mask_kind == ATTN_MASK_SLIDING_WINDOW) {
    if (!mp || mp->window < 0) return ATTN_ERR_ARG;
    p->mask.window = mp->window;
  }
  if (mask_kind == ATTN_MASK_DOCUMENT_CAUSAL) {
    if (!mp || !mp->doc_offsets || mp->n_docs < 1) return ATTN_ERR_ARG;
    if (Nq != Nkv) return ATTN_ERR_SHAPE;
    p->mask.doc = mp->doc_offsets;
    p->mask.n_docs = mp->n_docs;
  }
  return ATTN_OK;
}

// 3-D tensor map over a [BH, N, d] bf16 tensor: boxes of 64 elements (128 bytes,
// the 128-byte swizzle span) x box_rows rows x 1 head. Rows past N read as zeros.
attn_status make_map(CUtensorMap* map, const void* base, int BH, int N, int d,
                     unsigned box_rows = 128) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_LAUNCH;
}

attn_status from_cuda(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH; }

// Checked mode: the environment variable ATTN_CHECKED, set to anything but "" or "0"
// when the library first looks at it, makes every call with the document mask check
// its offsets on the device before its own kernels (a debugging aid: the table is
// otherwise trusted).
bool checked_mode() {
  static const bool on = [] {
    const char* e = std::getenv("ATTN_CHECKED");
    return e != nullptr && *e != '\0' && std::strcmp(e, "0") != 0;
  }();
  return on;
}

attn_status launch_doc_check(const int32_t* offs, int n_docs, int n, int* status,
                             cudaStream_t st) {
  constexpr int kThreadsPerBlock = 256;
  const long long blocks = ((long long)n_docs + kThreadsPerBlock) / kThreadsPerBlock;
  if (blocks > 0x7fffffffLL) return ATTN_ERR_SHAPE;
  doc_offsets_check_kernel<<<(int)blocks, kThreadsPerBlock, 0, st>>>(offs, n_docs, n, status);
  return from_cuda(cudaGetLastError());
}

attn_status maybe_check_docs(const Problem& p, const DeviceInfo* dev, cudaStream_t st) {
  if (p.mask.kind != ATTN_MASK_DOCUMENT_CAUSAL || !checked_mode()) return ATTN_OK;
  return launch_doc_check(p.mask.doc, p.mask.n_docs, p.mask.nq, dev->status, st);
}

attn_status fwd_common(bool simt, const void* q, const void* k, const void* v, void* o,
                       float* lse, int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale,
                       int mask_kind, const attn_mask_params* mp, int score_kind,
                       const attn_score_params* sp, void* stream) {
  Problem p;
  attn_status s = check_problem(B, Hq, Hkv, Nq, Nkv, d, scale, mask_kind, mp, score_kind, sp, &p);
  if (s != ATTN_OK) return s;
  if (simt && d == 256) return ATTN_ERR_SHAPE;
  // dropout: tensor-core path with d <= 128 only
  if ((score_kind & ATTN_SCORE_DROPOUT) && (simt || d == 256)) return ATTN_ERR_ARG;
  const long long rows_q = (long long)B * Hq * Nq;
  if (rows_q == 0) return ATTN_OK;
  if (!q || !o || !lse) return ATTN_ERR_ARG;
  if (Nkv > 0 && (!k || !v)) return ATTN_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_ALIGN;
  DeviceInfo* dev = nullptr;
  if ((s = current_device(&dev)) != ATTN_OK) return s;
  p.status = dev->status;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((s = maybe_check_docs(p, dev, st)) != ATTN_OK) return s;
  auto* ob = static_cast<__nv_bfloat16*>(o);
  if (Nkv == 0) return from_cuda(launch_fill_masked(rows_q, d, ob, lse, st));
  const auto* qb = static_cast<const __nv_bfloat16*>(q);
  const auto* kb = static_cast<const __nv_bfloat16*>(k);
  const auto* vb = static_cast<const __nv_bfloat16*>(v);
  if (simt) return from_cuda(launch_fwd_simt(p, qb, kb, vb, ob, lse, st));
  CUtensorMap tq, tk, tv;
  if (d == 256) {
    if ((s = make_map(&tk, k, B * Hkv, Nkv, d, 64)) != ATTN_OK) return s;
    if ((s = make_map(&tv, v, B * Hkv, Nkv, d, 64)) != ATTN_OK) return s;
    return from_cuda(launch_fwd256_tc(p, qb, tk, tv, ob, lse, st));
  }
  if ((s = make_map(&tq, q, B * Hq, Nq, d)) != ATTN_OK) return s;
  if ((s = make_map(&tk, k, B * Hkv, Nkv, d)) != ATTN_OK) return s;
  if ((s = make_map(&tv, v, B * Hkv, Nkv, d)) != ATTN_OK) return s;
  return from_cuda(launch_fwd_tc(p, tq, tk, tv, ob, lse, st));
}

// Workspace of the backward: the three row-term arrays of RowTerms, each starting on
// a 256-byte boundary. rows = B * Hq * nq_pad.
size_t row_terms_bytes(long long rows, int nq_pad) {
  return 2 * round256((size_t)rows * sizeof(float)) + round256((size_t)nq_pad * sizeof(int));
}
RowTerms row_terms(int B, int Hq, int nq_pad, void* workspace) {
  const size_t plane = round256((size_t)B * Hq * nq_pad * sizeof(float));
  uint8_t* base = static_cast<uint8_t*>(workspace);
  return RowTerms{reinterpret_cast<float*>(base), reinterpret_cast<float*>(base + plane),
                  reinterpret_cast<int*>(base + 2 * plane)};
}

attn_status bwd_common(bool simt, const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                       int Hq, int Hkv, int Nq, int Nkv, int d, float scale, int mask_kind,
                       const attn_mask_params* mp, int score_kind, const attn_score_params* sp,
                       void* workspace, size_t workspace_bytes, void* stream,
                       int phases = ATTN_BWD_ALL) {
  if (phases & ~ATTN_BWD_ALL) return ATTN_ERR_ARG;
  Problem p;
  attn_status s = check_problem(B, Hq, Hkv, Nq, Nkv, d, scale, mask_kind, mp, score_kind, sp, &p);
  if (s != ATTN_OK) return s;
  if (simt && d == 256) return ATTN_ERR_SHAPE;  // the SIMT backward: d = 64 and 128
  // dropout: tensor-core path with d <= 128 only (like the forward)
  if ((score_kind & ATTN_SCORE_DROPOUT) && (simt || d == 256)) return ATTN_ERR_ARG;
  const long long rows_q = (long long)B * Hq * Nq, rows_k = (long long)B * Hkv * Nkv;
  if (rows_q == 0 && rows_k == 0) return ATTN_OK;
  if (rows_q > 0 && (!q || !o || !lse || !dout || !dq)) return ATTN_ERR_ARG;
  if (rows_k > 0 && (!k || !v || !dk || !dv)) return ATTN_ERR_ARG;
  const void* ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv};
  for (const void* ptr : ptrs)
    if (!aligned16(ptr)) return ATTN_ERR_ALIGN;
  const size_t need = attn_bwd_workspace_size(B, Hq, Hkv, Nq, Nkv, d);
  if (need > 0 && (!workspace || workspace_bytes < need)) return ATTN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_ALIGN;
  DeviceInfo* dev = nullptr;
  if ((s = current_device(&dev)) != ATTN_OK) return s;
  p.status = dev->status;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((s = maybe_check_docs(p, dev, st)) != ATTN_OK) return s;
  // With no queries nothing reaches the keys, and with no keys nothing reaches the
  // queries: those gradients are zero.
  if (rows_q == 0 || rows_k == 0) {
    const bool zq = rows_q > 0 && (phases & ATTN_BWD_DQ);
    const bool zk = rows_k > 0 && (phases & ATTN_BWD_DKDV);
    if (zq && cudaMemsetAsync(dq, 0, (size_t)rows_q * d * 2, st) != cudaSuccess)
      return ATTN_ERR_LAUNCH;
    if (zk && cudaMemsetAsync(dk, 0, (size_t)rows_k * d * 2, st) != cudaSuccess)
      return ATTN_ERR_LAUNCH;
    if (zk && cudaMemsetAsync(dv, 0, (size_t)rows_k * d * 2, st) != cudaSuccess)
      return ATTN_ERR_LAUNCH;
    return ATTN_OK;
  }
  const RowTerms rt = row_terms(B, Hq, p.nq_pad, workspace);
  const auto* qb = static_cast<const __nv_bfloat16*>(q);
  const auto* kb = static_cast<const __nv_bfloat16*>(k);
  const auto* vb = static_cast<const __nv_bfloat16*>(v);
  const auto* dob = static_cast<const __nv_bfloat16*>(dout);
  auto* dqb = static_cast<__nv_bfloat16*>(dq);
  auto* dkb = static_cast<__nv_bfloat16*>(dk);
  auto* dvb = static_cast<__nv_bfloat16*>(dv);
  BwdMaps maps;  // built before the first launch: errors launch nothing
  if (!simt && (phases & (ATTN_BWD_DKDV | ATTN_BWD_DQ))) {
    // 128-row boxes for the tiles a CTA loads once, 64-row boxes for the streamed ones
    if ((s = make_map(&maps.v128, v, B * Hkv, Nkv, d)) != ATTN_OK) return s;
    if ((s = make_map(&maps.q64, q, B * Hq, Nq, d, 64)) != ATTN_OK) return s;
    if ((s = make_map(&maps.do64, dout, B * Hq, Nq, d, 64)) != ATTN_OK) return s;
    if ((s = make_map(&maps.k64, k, B * Hkv, Nkv, d, 64)) != ATTN_OK) return s;
    if ((s = make_map(&maps.v64, v, B * Hkv, Nkv, d, 64)) != ATTN_OK) return s;
    if ((s = make_map(&maps.do128, dout, B * Hq, Nq, d)) != ATTN_OK) return s;
    if (d <= 128 && (s = make_map(&maps.k128, k, B * Hkv, Nkv, d)) != ATTN_OK) return s;
    if (d <= 128 && (s = make_map(&maps.q128, q, B * Hq, Nq, d)) != ATTN_OK) return s;
  }
  if ((phases & ATTN_BWD_ROWDOT) &&
      (s = from_cuda(launch_bwd_rowdot(p, static_cast<const __nv_bfloat16*>(o), dob, lse, rt,
                                       st))) != ATTN_OK)
    return s;
  if (simt) {
    if ((phases & (ATTN_BWD_DKDV | ATTN_BWD_DQ)) != (ATTN_BWD_DKDV | ATTN_BWD_DQ))
      return phases & (ATTN_BWD_DKDV | ATTN_BWD_DQ) ? ATTN_ERR_ARG : ATTN_OK;
    return from_cuda(launch_bwd_simt(p, qb, kb, vb, lse, dob, rt.delta, dqb, dkb, dvb, st));
  }
  if (!(phases & (ATTN_BWD_DKDV | ATTN_BWD_DQ))) return ATTN_OK;
  const bool run_kv = (phases & ATTN_BWD_DKDV) != 0, run_q = (phases & ATTN_BWD_DQ) != 0;
  if (d == 256)
    return from_cuda(launch_bwd256_tc(p, maps, rt, qb, dob, kb, dqb, dkb, dvb, run_kv, run_q, st));
  return from_cuda(
      launch_bwd_tc(p, maps, rt, qb, dob, kb, vb, dqb, dkb, dvb, run_kv, run_q, st));
}

// ---------------------------------------------------------------- static workspace
// Scratch of attn_bwd_static_workspace: the backward's row terms (three 4-byte words
// per padded query row) for callers that cannot allocate. One copy per device, shared
// by every call on that device.
constexpr size_t kStaticWords = 3 * (size_t)ATTN_STATIC_WORKSPACE_ROWS;
static __device__ __align__(256) float g_static_workspace[kStaticWords];

std::mutex g_static_mu;
float* g_static_ptr[kMaxDevices];  // device address of g_static_workspace, per device

// Device address of g_static_workspace on the current device. The host-side name
// of the array is only a stand-in for it, so the address is looked up once per
// device, with that device current, and cached.
attn_status static_workspace_ptr(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess || ptr == nullptr)
      return ATTN_ERR_LAUNCH;
    g_static_ptr[dev] = static_cast<float*>(ptr);
  }
  *out = g_static_ptr[dev];
  return ATTN_OK;
}

// ---------------------------------------------------------------- FP8
// Tensor map over bytes [dz][dy][dx] with rows of row_bytes, box 128 x 128 x 1,
// 128-byte swizzle (e4m3 tiles: 128 values of the innermost dimension per row).
attn_status make_map8(CUtensorMap* map, const void* base, int dx, int dy, int dz,
                      size_t row_bytes) {
  cuuint64_t dims[3] = {(cuuint64_t)dx, (cuuint64_t)dy, (cuuint64_t)dz};
  cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)row_bytes * dy};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_LAUNCH;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// ---------------------------------------------------------------- paged decode
// Page sizes whose 64-key tiles never straddle a page: 8, 16, 32 (several pages per
// tile) or any multiple of 64.
bool decode_page_size_ok(int ps) { return ps == 8 || ps == 16 || ps == 32 || (ps > 0 && ps % 64 == 0); }

long long decode_chunks(int max_seq_len, int split_keys) {
  return max_seq_len <= 0 ? 1 : ((long long)max_seq_len + split_keys - 1) / split_keys;
}

// Split-mode scratch: L2 of every (chunk, row), then O of every (chunk, row).
size_t decode_lse_plane(long long n_chunks, long long rows) {
  return round256((size_t)(n_chunks * rows) * sizeof(float));
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int Hq, int Hkv, int Nq, int Nkv, int d, float scale, int mask_kind,
                     const attn_mask_params* mask_params, int score_kind,
                     const attn_score_params* score_params, void* stream) {
  return fwd_common(false, q, k, v, o, lse, B, Hq, Hkv, Nq, Nkv, d, scale, mask_kind,
                    mask_params, score_kind, score_params, stream);
}

attn_status attn_fwd_simt(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale,
                          int mask_kind, const attn_mask_params* mask_params, int score_kind,
                          const attn_score_params* score_params, void* stream) {
  return fwd_common(true, q, k, v, o, lse, B, Hq, Hkv, Nq, Nkv, d, scale, mask_kind,
                    mask_params, score_kind, score_params, stream);
}

size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int Nq, int Nkv, int d) {
  (void)Hkv; (void)Nkv; (void)d;
  if (B <= 0 || Hq <= 0 || Nq <= 0) return 0;
  const int nq_pad = (int)(((long long)Nq + 127) / 128 * 128);
  return row_terms_bytes((long long)B * Hq * nq_pad, nq_pad);
}

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                     int Hq, int Hkv, int Nq, int Nkv, int d, float scale, int mask_kind,
                     const attn_mask_params* mask_params, int score_kind,
                     const attn_score_params* score_params, void* workspace,
                     size_t workspace_bytes, void* stream) {
  return bwd_common(false, q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Nq, Nkv, d, scale,
                    mask_kind, mask_params, score_kind, score_params, workspace,
                    workspace_bytes, stream);
}

attn_status attn_bwd_simt(const void* q, const void* k, const void* v, const void* o,
                          const float* lse, const void* dout, void* dq, void* dk, void* dv,
                          int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale,
                          int mask_kind, const attn_mask_params* mask_params, int score_kind,
                          const attn_score_params* score_params, void* workspace,
                          size_t workspace_bytes, void* stream) {
  return bwd_common(true, q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Nq, Nkv, d, scale,
                    mask_kind, mask_params, score_kind, score_params, workspace,
                    workspace_bytes, stream);
}

attn_status attn_bwd_phases(int phases, const void* q, const void* k, const void* v,
                            const void* o, const float* lse, const void* dout, void* dq,
                            void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                            float scale, int mask_kind, const attn_mask_params* mask_params,
                            int score_kind, const attn_score_params* score_params,
                            void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_common(false, q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Nq, Nkv, d, scale,
                    mask_kind, mask_params, score_kind, score_params, workspace,
                    workspace_bytes, stream, phases);
}

attn_status attn_bwd_static_workspace(const void* q, const void* k, const void* v,
                                      const void* o, const float* lse, const void* dout,
                                      void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                                      int Nq, int Nkv, int d, float scale, int mask_kind,
                                      const attn_mask_params* mask_params, int score_kind,
                                      const attn_score_params* score_params, void* stream) {
  if (B < 0 || Hq < 0 || Nq < 0) return ATTN_ERR_SHAPE;
  const long long rows = (long long)B * Hq * ((Nq + 127LL) / 128 * 128);
  if (rows > ATTN_STATIC_WORKSPACE_ROWS) return ATTN_ERR_WORKSPACE;
  float* ws = nullptr;
  if (rows > 0) {
    DeviceInfo* dev = nullptr;
    attn_status s = current_device(&dev);  // rejects devices other than sm_103 first
    if (s != ATTN_OK) return s;
    if ((s = static_workspace_ptr(&ws)) != ATTN_OK) return s;
  }
  return bwd_common(false, q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Nq, Nkv, d, scale,
                    mask_kind, mask_params, score_kind, score_params, ws,
                    ws ? kStaticWords * sizeof(float) : 0, stream);
}

size_t attn_fp8_v_row_bytes(int Nkv) { return Nkv <= 0 ? 0 : (size_t)(Nkv + 15) / 16 * 16; }

attn_status attn_quantize_fp8(const void* x, void* out, float* scales, int BH, int N, int d,
                              int layout, void* stream) {
  if (BH < 0 || N < 0 || (d != 64 && d != 128)) return ATTN_ERR_SHAPE;
  if (layout != ATTN_FP8_TILES && layout != ATTN_FP8_V_TRANSPOSED) return ATTN_ERR_ARG;
  if ((long long)BH * N == 0 && layout == ATTN_FP8_TILES) return ATTN_OK;
  if (BH == 0) return ATTN_OK;
  if (!out || !scales || (N > 0 && !x)) return ATTN_ERR_ARG;
  if (!aligned16(x) || !aligned16(out) || !aligned4(scales)) return ATTN_ERR_ALIGN;
  if (layout == ATTN_FP8_TILES && BH > 65535) return ATTN_ERR_SHAPE;
  DeviceInfo* dev = nullptr;
  attn_status s = current_device(&dev);
  if (s != ATTN_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  auto* ob = static_cast<uint8_t*>(out);
  if (layout == ATTN_FP8_TILES) return from_cuda(launch_quantize_tiles(xb, ob, scales, BH, N, d, st));
  return from_cuda(launch_quantize_v_transposed(xb, ob, scales, BH, N, d, st));
}

attn_status attn_fwd_fp8(const void* q8, const void* k8, const void* v8t, const float* q_scale,
                         const float* k_scale, const float* v_scale, void* o, float* lse, int B,
                         int Hq, int Hkv, int Nq, int Nkv, int d, float scale, int mask_kind,
                         const attn_mask_params* mask_params, int score_kind,
                         const attn_score_params* score_params, void* stream) {
  Problem p;
  attn_status s = check_problem(B, Hq, Hkv, Nq, Nkv, d, scale, mask_kind, mask_params,
                                score_kind, score_params, &p);
  if (s != ATTN_OK) return s;
  if (d != 128) return ATTN_ERR_SHAPE;  // FP8 forward: d = 128
  if (score_kind & ATTN_SCORE_DROPOUT) return ATTN_ERR_ARG;
  const long long rows_q = (long long)B * Hq * Nq;
  if (rows_q == 0) return ATTN_OK;
  if (!q8 || !q_scale || !o || !lse) return ATTN_ERR_ARG;
  if (Nkv > 0 && (!k8 || !v8t || !k_scale || !v_scale)) return ATTN_ERR_ARG;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8t) || !aligned16(o) || !aligned16(lse) ||
      !aligned4(q_scale) || !aligned4(k_scale) || !aligned4(v_scale))
    return ATTN_ERR_ALIGN;
  DeviceInfo* dev = nullptr;
  if ((s = current_device(&dev)) != ATTN_OK) return s;
  p.status = dev->status;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((s = maybe_check_docs(p, dev, st)) != ATTN_OK) return s;
  auto* ob = static_cast<__nv_bfloat16*>(o);
  if (Nkv == 0) return from_cuda(launch_fill_masked(rows_q, d, ob, lse, st));
  CUtensorMap tq, tk, tvt;
  if ((s = make_map8(&tq, q8, d, Nq, B * Hq, d)) != ATTN_OK) return s;
  if ((s = make_map8(&tk, k8, d, Nkv, B * Hkv, d)) != ATTN_OK) return s;
  if ((s = make_map8(&tvt, v8t, Nkv, d, B * Hkv, attn_fp8_v_row_bytes(Nkv))) != ATTN_OK) return s;
  return from_cuda(launch_fwd_fp8_tc(p, tq, tk, tvt, q_scale, k_scale, v_scale, ob, lse, st));
}

int attn_decode_split_keys(int B, int Hq, int Hkv, int Nq, long long total_kv_tokens,
                           int num_sms) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || total_kv_tokens <= 0 || Hq % Hkv != 0)
    return 256;
  const long long rows = (long long)(Hq / Hkv) * Nq;
  const long long row_tiles = (rows + 63) / 64;
  // about ten work items per SM for the persistent kernel (one CTA per SM)
  const long long target = 10LL * (num_sms > 0 ? num_sms : 148);
  const long long work = total_kv_tokens * Hkv * row_tiles;
  long long keys = (work + target - 1) / target;
  keys = (keys + 63) / 64 * 64;
  if (keys < 256) keys = 256;
  if (keys > (1 << 24)) keys = 1 << 24;
  return (int)keys;
}

size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int Nq, int d, int max_seq_len,
                                  int split_keys) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || d <= 0 || split_keys <= 0 || Hq % Hkv != 0)
    return 0;
  const long long copies = decode_row_copies((int)std::min<long long>((long long)(Hq / Hkv) * Nq, 1 << 30));
  const long long n = decode_chunks(max_seq_len, split_keys) * copies;
  if (n <= 1 || max_seq_len <= 0) return 0;
  const long long rows = (long long)B * Hq * Nq;
  return decode_lse_plane(n, rows) + round256((size_t)(n * rows) * d * sizeof(float));
}

attn_status attn_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* page_table, const int32_t* seq_lens, void* o,
                              float* lse, int B, int Hq, int Hkv, int Nq, int d, int num_pages,
                              int page_size, int max_pages_per_seq, int max_seq_len,
                              int split_keys, float scale, int mask_kind,
                              const attn_mask_params* mask_params, int score_kind,
                              const attn_score_params* score_params, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (B < 0 || Hq < 0 || Hkv < 0 || Nq < 0 || num_pages < 0 || max_pages_per_seq < 0 ||
      max_seq_len < 0)
    return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128) return ATTN_ERR_SHAPE;
  if (Hkv == 0 ? Hq != 0 : (Hq % Hkv) != 0) return ATTN_ERR_SHAPE;
  if (!decode_page_size_ok(page_size)) return ATTN_ERR_SHAPE;
  if ((long long)max_seq_len > (long long)max_pages_per_seq * page_size) return ATTN_ERR_SHAPE;
  if (split_keys <= 0 || split_keys % 64 != 0) return ATTN_ERR_ARG;
  if (!std::isfinite(scale)) return ATTN_ERR_ARG;
  if (mask_kind != ATTN_MASK_NONE && mask_kind != ATTN_MASK_CAUSAL &&
      mask_kind != ATTN_MASK_SLIDING_WINDOW)
    return ATTN_ERR_ARG;
  if (score_kind & ~(ATTN_SCORE_ALIBI | ATTN_SCORE_SOFTCAP)) return ATTN_ERR_ARG;
  DecodeProblem p{};
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.Nq = Nq; p.d = d;
  p.page_size = page_size; p.max_pages = max_pages_per_seq; p.num_pages = num_pages;
  p.max_seq_len = max_seq_len;
  p.chunk = split_keys;
  p.scale = scale;
  p.score_kind = score_kind;
  p.mask_kind = mask_kind;
  if (score_kind & ATTN_SCORE_SOFTCAP) {
    if (!score_params || !(score_params->softcap > 0.f) || !std::isfinite(score_params->softcap))
      return ATTN_ERR_ARG;
    p.softcap = score_params->softcap;
  }
  if (mask_kind == ATTN_MASK_SLIDING_WINDOW) {
    if (!mask_params || mask_params->window < 0) return ATTN_ERR_ARG;
    p.window = mask_params->window;
  }
  const long long rows_total = (long long)B * Hq * Nq;
  if (rows_total == 0) return ATTN_OK;
  const long long n_chunks = decode_chunks(max_seq_len, split_keys);
  const long long row_tiles = ((long long)(Hq / Hkv) * Nq + 63) / 64;
  if (rows_total > 0x7fffffffLL || (long long)B * Hkv * row_tiles * n_chunks > (1LL << 40) ||
      (long long)num_pages * Hkv * page_size > 0x7fffffffLL || n_chunks > 0x7fffffffLL)
    return ATTN_ERR_SHAPE;
  p.n_chunks = (int)n_chunks;
  if (!q || !o || !lse || !seq_lens) return ATTN_ERR_ARG;
  if (max_seq_len > 0 && (!k_cache || !v_cache || !page_table || num_pages == 0))
    return ATTN_ERR_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
      !aligned16(lse) || !aligned4(page_table) || !aligned4(seq_lens))
    return ATTN_ERR_ALIGN;
  const size_t need = attn_decode_workspace_size(B, Hq, Hkv, Nq, d, max_seq_len, split_keys);
  if (need > 0 && (!workspace || workspace_bytes < need)) return ATTN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_ALIGN;
  DeviceInfo* dev = nullptr;
  attn_status s = current_device(&dev);
  if (s != ATTN_OK) return s;
  p.status = dev->status;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto* ob = static_cast<__nv_bfloat16*>(o);
  if (max_seq_len == 0) return from_cuda(launch_fill_masked(rows_total, d, ob, lse, st));
  DecodeOut out{ob, lse, nullptr, nullptr};
  if (need > 0) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    out.part_lse = reinterpret_cast<float*>(ws);
    const long long parts =
        n_chunks * decode_row_copies((int)std::min<long long>((long long)(Hq / Hkv) * Nq, 1 << 30));
    out.part_o = reinterpret_cast<float*>(ws + decode_lse_plane(parts, rows_total));
  }
  CUtensorMap tk, tv;
  const int kv_rows = num_pages * Hkv * page_size;
  const unsigned box = page_size < 64 ? (unsigned)page_size : 64u;
  if ((s = make_map(&tk, k_cache, 1, kv_rows, d, box)) != ATTN_OK) return s;
  if ((s = make_map(&tv, v_cache, 1, kv_rows, d, box)) != ATTN_OK) return s;
  p.q = static_cast<const __nv_bfloat16*>(q);
  return from_cuda(launch_decode_tc(p, tk, tv, out, dev->num_sms, st));
}

attn_status attn_classify_tiles(int mask_kind, const attn_mask_params* mask_params, int Nq,
                                int Nkv, int32_t* classes, void* stream) {
  Problem p;
  attn_status s = check_problem(1, 1, 1, Nq, Nkv, 64, 1.0f, mask_kind, mask_params, 0, nullptr,
                                &p);
  if (s != ATTN_OK) return s;
  if (Nq == 0 || Nkv == 0) return ATTN_OK;
  if (!classes) return ATTN_ERR_ARG;
  DeviceInfo* dev = nullptr;
  if ((s = current_device(&dev)) != ATTN_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((s = maybe_check_docs(p, dev, st)) != ATTN_OK) return s;
  return from_cuda(launch_classify(p.mask, classes, st));
}

attn_status attn_check_doc_offsets(const int32_t* doc_offsets, int n_docs, int N,
                                   void* stream) {
  if (!doc_offsets || n_docs < 1 || N < 0) return ATTN_ERR_ARG;
  if (!aligned4(doc_offsets)) return ATTN_ERR_ALIGN;
  DeviceInfo* dev = nullptr;
  attn_status s = current_device(&dev);
  if (s != ATTN_OK) return s;
  return launch_doc_check(doc_offsets, n_docs, N, dev->status, static_cast<cudaStream_t>(stream));
}

attn_status attn_selftest_wait_timeout(void* stream) {
  DeviceInfo* dev = nullptr;
  attn_status s = current_device(&dev);
  if (s != ATTN_OK) return s;
  attn::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev->status);
  return from_cuda(cudaGetLastError());
}

attn_status attn_device_status(void* stream) {
  DeviceInfo* dev = nullptr;
  attn_status s = current_device(&dev);
  if (s != ATTN_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return ATTN_ERR_LAUNCH;
  int value = 0;
  if (cudaMemcpy(&value, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  if (value != 0) {
    const int zero = 0;
    if (cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return ATTN_ERR_LAUNCH;
    return (value & DEV_TIMEOUT_BIT) ? ATTN_ERR_DEVICE_TIMEOUT : ATTN_ERR_DEVICE_INPUT;
  }
  return ATTN_OK;
}

const char* attn_strerror(attn_status status) {
  switch (status) {
    case ATTN_OK: return "success";
    case ATTN_ERR_ARG: return "invalid argument (null pointer, unknown kind or bad parameter)";
    case ATTN_ERR_SHAPE:
      return "unsupported shape (d must be 64 or 128, or 256 for attn_fwd; Hq a multiple of Hkv)";
    case ATTN_ERR_ALIGN: return "tensor pointer not 16-byte aligned";
    case ATTN_ERR_ARCH: return "current device is not an sm_103 (GB300) GPU";
    case ATTN_ERR_WORKSPACE: return "workspace missing or smaller than attn_bwd_workspace_size";
    case ATTN_ERR_LAUNCH: return "CUDA launch or driver call failed";
    case ATTN_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait";
    case ATTN_ERR_DEVICE_INPUT:
      return "a kernel met an out-of-range device input (sequence length or page index)";
  }
  return "unknown status";
}

}  // extern "C"
