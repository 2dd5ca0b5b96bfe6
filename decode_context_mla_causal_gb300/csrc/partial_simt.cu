// Step 3 (first version): split-KV absorbed-MLA partial attention on CUDA cores.
//
// "[ROCm][MLA][DCP] Support causal multi-token verification", Implementation
// item 3: per rank, attention over that rank's local KV emitting unreduced
// partial outputs with base-2 max/sum statistics. One CTA per
// (16 query rows, split, rank x sequence). Keys arrive 32 tokens at a time,
// dequantised to fp32 in shared memory; each warp scores two rows against the
// chunk, keeps an online base-2 softmax, and all threads accumulate P.V.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace dcpmla {
namespace {

constexpr int kRows = 16;
constexpr int kTok = 32;
constexpr int kThreads = 256;
constexpr int kKStride = kDqk + 1;  // padded fp32 row: conflict-free column reads
constexpr float kLog2e = 1.4426950408889634f;

constexpr size_t kSmemBytes =
    sizeof(float) * (kRows * kDqk + kTok * kKStride + kRows * kTok + kRows * 4) +
    sizeof(int64_t) * kTok + sizeof(int) * (kRows + 4);

template <bool kFp8>
__device__ __forceinline__ void load_row_chunk(const uint8_t* row_bytes, int e, float* dst) {
  // 4 consecutive elements starting at element e
  if (kFp8) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(row_bytes + e);
    __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFF), __NV_E4M3);
    __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
    float2 a = __half22float2(*reinterpret_cast<__half2*>(&lo));
    float2 b = __half22float2(*reinterpret_cast<__half2*>(&hi));
    dst[0] = a.x;
    dst[1] = a.y;
    dst[2] = b.x;
    dst[3] = b.y;
  } else {
    const uint2 w = *reinterpret_cast<const uint2*>(row_bytes + 2 * e);
    dst[0] = __uint_as_float(w.x << 16);
    dst[1] = __uint_as_float(w.x & 0xFFFF0000u);
    dst[2] = __uint_as_float(w.y << 16);
    dst[3] = __uint_as_float(w.y & 0xFFFF0000u);
  }
}

template <bool kFp8>
__global__ void __launch_bounds__(kThreads)
partial_simt_kernel(int batch, int qlen, int H, int num_splits, int subpage, int max_pages,
                    int64_t pool_rows, const __nv_bfloat16* __restrict__ q,
                    const uint8_t* __restrict__ kv, const float* __restrict__ kv_scale_ptr,
                    float softmax_scale, const int32_t* __restrict__ row_len,
                    const int32_t* __restrict__ page_ids, const int32_t* __restrict__ split_beg,
                    const int32_t* __restrict__ split_end, float* __restrict__ part_o,
                    float* __restrict__ part_m, float* __restrict__ part_l, uint32_t* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* Qs = reinterpret_cast<float*>(smem_raw);
  float* Ks = Qs + kRows * kDqk;
  float* Ps = Ks + kTok * kKStride;
  float* s_alpha = Ps + kRows * kTok;
  float* s_m = s_alpha + kRows;
  float* s_l = s_m + kRows;
  int64_t* s_rowoff = reinterpret_cast<int64_t*>(s_l + 2 * kRows);
  int* s_lim = reinterpret_cast<int*>(s_rowoff + kTok);
  int* s_misc = s_lim + kRows;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int b = blockIdx.z % batch;
  const int k = blockIdx.z / batch;
  const int s = blockIdx.y;
  const int qrows = qlen * H;
  const int qr0 = blockIdx.x * kRows;
  const int R = batch * qlen;
  const float kv_scale = kv_scale_ptr ? *kv_scale_ptr : 1.0f;
  const float sc = softmax_scale * kv_scale * kLog2e;
  const size_t elem = kFp8 ? 1 : 2;
  const uint8_t* pool = kv + (size_t)k * pool_rows * kDqk * elem;

  if (tid < kRows) {
    const int qr = qr0 + tid;
    int lim = 0;
    if (qr < qrows) lim = row_len[(int64_t)k * R + (int64_t)b * qlen + qr / H];
    s_lim[tid] = lim;
  }
  if (tid == 0) {
    const int64_t sb = ((int64_t)k * batch + b) * num_splits + s;
    int beg = split_beg[sb], end = split_end[sb];
    if (beg < 0 || end < beg || end > max_pages) {
      raise_status(status, DCP_STATUS_BAD_SPLIT);
      beg = end = 0;
    }
    s_misc[0] = beg;
    s_misc[1] = end;
  }
  // q rows of this CTA, bf16 -> fp32
  for (int i = tid; i < kRows * kDqk; i += kThreads) {
    const int r = i / kDqk, d = i % kDqk;
    const int qr = qr0 + r;
    float v = 0.f;
    if (qr < qrows) v = __bfloat162float(q[((int64_t)b * qrows + qr) * kDqk + d]);
    Qs[i] = v;
  }
  __syncthreads();
  int top = 0;
  for (int i = 0; i < kRows; ++i) top = max(top, s_lim[i]);
  const int t0 = s_misc[0] * subpage;
  const int t1 = min(s_misc[1] * subpage, top);
  const int32_t* pages = page_ids + ((int64_t)k * batch + b) * max_pages;
  const int64_t num_pages_pool = pool_rows / subpage;

  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.f;
  const int prow = tid / 16;
  const int pd0 = tid % 16;

  for (int c = t0; c < t1; c += kTok) {
    if (tid < kTok) {
      const int li = c + tid;
      int64_t off = -1;
      if (li < t1) {
        const int32_t pg = pages[li / subpage];
        if (pg >= 0 && pg < num_pages_pool) {
          off = ((int64_t)pg * subpage + li % subpage) * kDqk * elem;
        } else {
          raise_status(status, DCP_STATUS_BAD_PAGE);
        }
      }
      s_rowoff[tid] = off;
    }
    __syncthreads();
    for (int i = tid; i < kTok * (kDqk / 4); i += kThreads) {
      const int tk = i / (kDqk / 4);
      const int e = (i % (kDqk / 4)) * 4;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      const int64_t off = s_rowoff[tk];
      if (off >= 0) load_row_chunk<kFp8>(pool + off, e, v);
      float* dst = Ks + tk * kKStride + e;
      dst[0] = v[0];
      dst[1] = v[1];
      dst[2] = v[2];
      dst[3] = v[3];
    }
    __syncthreads();
    // scores: warp w owns rows 2w, 2w+1; lane = token
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int r = warp * 2 + rr;
      const float* qv = Qs + r * kDqk;
      const float* kvr = Ks + lane * kKStride;
      float dot = 0.f;
#pragma unroll 8
      for (int d = 0; d < kDqk; ++d) dot = fmaf(qv[d], kvr[d], dot);
      const int li = c + lane;
      const bool ok = li < t1 && li < s_lim[r] && s_rowoff[lane] >= 0;
      const float sv = ok ? dot * sc : -INFINITY;
      float cm = sv;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
      const float m_new = fmaxf(m_run[rr], cm);
      float p = 0.f, alpha = 1.f;
      if (m_new != -INFINITY) {
        p = ok ? exp2f(sv - m_new) : 0.f;
        alpha = m_run[rr] == -INFINITY ? 0.f : exp2f(m_run[rr] - m_new);
      }
      float ps = p;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l_run[rr] = l_run[rr] * alpha + ps;
      m_run[rr] = m_new;
      Ps[r * kTok + lane] = p;
      if (lane == 0) s_alpha[r] = alpha;
    }
    __syncthreads();
    {
      const float a = s_alpha[prow];
      const float* pr = Ps + prow * kTok;
#pragma unroll
      for (int kk = 0; kk < 32; ++kk) {
        const int d = pd0 + 16 * kk;
        float sum = 0.f;
#pragma unroll 8
        for (int tk = 0; tk < kTok; ++tk) sum = fmaf(pr[tk], Ks[tk * kKStride + d], sum);
        acc[kk] = fmaf(acc[kk], a, sum);
      }
    }
    __syncthreads();
  }
  if (lane == 0) {
    s_m[warp * 2] = m_run[0];
    s_m[warp * 2 + 1] = m_run[1];
    s_l[warp * 2] = l_run[0];
    s_l[warp * 2 + 1] = l_run[1];
  }
  __syncthreads();
  const int qr = qr0 + prow;
  if (qr < qrows) {
    const int64_t rh = (int64_t)b * qrows + qr;  // (b*qlen + j)*H + h
    const int64_t base = ((int64_t)k * num_splits + s) * ((int64_t)R * H) + rh;
    const float l = s_l[prow];
    const float inv = l > 0.f ? kv_scale / l : 0.f;
    float* dst = part_o + base * kDv;
#pragma unroll
    for (int kk = 0; kk < 32; ++kk) dst[pd0 + 16 * kk] = acc[kk] * inv;
    if (pd0 == 0) {
      part_m[base] = l > 0.f ? s_m[prow] : -INFINITY;
      part_l[base] = l;
    }
  }
}

}  // namespace

cudaError_t launch_partial_simt(const dcp_mla_dims& d, const Derived& x, const void* q,
                           const void* kv, dcp_kv_dtype kv_dtype, const float* kv_scale,
                           float softmax_scale, int num_ranks, const int32_t* row_len,
                           const int32_t* page_ids, const int32_t* split_beg,
                           const int32_t* split_end, float* part_o, float* part_m,
                           float* part_l, uint32_t* status, cudaStream_t stream) {
  const int qrows = d.qlen * d.num_heads;
  dim3 grid((qrows + kRows - 1) / kRows, d.num_splits, num_ranks * d.batch);
  if (grid.y > 65535 || grid.z > 65535) return cudaErrorInvalidConfiguration;
  const int64_t pool_rows = (int64_t)d.num_blocks * d.block_size;
  const bool fp8 = kv_dtype == DCP_KV_FP8_E4M3;
  auto kern = fp8 ? partial_simt_kernel<true> : partial_simt_kernel<false>;
  // The shared-memory opt-in is a per-device function attribute: set it once per
  // device (before any stream capture, since the first call does it).
  static bool attr_set[2][64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[fp8][dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[fp8][dev] = true;
  }
  kern<<<grid, kThreads, kSmemBytes, stream>>>(
      d.batch, d.qlen, d.num_heads, d.num_splits, x.subpage, x.max_pages, pool_rows,
      reinterpret_cast<const __nv_bfloat16*>(q), reinterpret_cast<const uint8_t*>(kv), kv_scale,
      softmax_scale, row_len, page_ids, split_beg, split_end, part_o, part_m, part_l, status);
  return cudaGetLastError();
}

}  // namespace dcpmla
