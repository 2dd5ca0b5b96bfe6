// Step 4: LSE merge of every split of every rank into the BF16 output.
//
// "Context Parallel Guide (PCP & DCP)", Decode: the per-rank partial outputs
// are LSE-corrected and summed. "[ROCm][MLA][DCP] Support causal multi-token
// verification", Implementation item 3: base-2 partial statistics become a BF16
// output plus a natural-log LSE. Splits and ranks are merged in one pass: with
// m, l, o per (rank, split), M = max m, w = 2^(m - M) * l,
// O = sum w*o / sum w, LSE = (M + log2 sum w) * ln 2 (M kept as a running maximum).
//
// HBM-bound, two forms:
//   merge_all_kernel   every split slot is expected to hold work (no wave balancing):
//                      one CTA per (row, head), 4 dims per thread; a batch of four
//                      partials' m, l and output loads are in flight together.
//   merge_live_kernel  wave balancing leaves most slots empty: one warp per (row,
//                      head), 16 dims per lane; the m and l of 32 partials come in one
//                      load per lane, a ballot lists the live ones (m finite, l > 0;
//                      empty splits and slots the partial kernel skipped are -inf),
//                      and only their outputs are read, four at a time.
// Both write 1 KB of BF16 per (row, head).
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"

namespace dcpmla {
namespace {

constexpr int kMergeThreads = 128;  // merge_all_kernel: 4 dims per thread
constexpr int kBatch = 4;           // partials whose loads are issued together
constexpr int kLiveWarps = 8;       // merge_live_kernel: entries per CTA
constexpr float kLn2 = 0.6931471805599453f;

// Per-rank LSE of entry rh over its splits (natural log), one rank per thread.
__device__ __forceinline__ void write_rank_lse(int rh, int rows_heads, int num_ranks,
                                               int num_splits, const float* part_m,
                                               const float* part_l, float* rank_lse, int first,
                                               int step) {
  for (int k = first; k < num_ranks; k += step) {
    float Mk = -INFINITY;
    for (int s = 0; s < num_splits; ++s)
      Mk = fmaxf(Mk, part_m[((int64_t)k * num_splits + s) * rows_heads + rh]);
    float dk = 0.f;
    if (Mk != -INFINITY) {
      for (int s = 0; s < num_splits; ++s) {
        const int64_t idx = ((int64_t)k * num_splits + s) * rows_heads + rh;
        const float m = part_m[idx];
        const float l = part_l[idx];
        if (m != -INFINITY && l > 0.f) dk += exp2f(m - Mk) * l;
      }
    }
    rank_lse[(int64_t)k * rows_heads + rh] = dk > 0.f ? (Mk + log2f(dk)) * kLn2 : -INFINITY;
  }
}

__global__ void __launch_bounds__(kMergeThreads)
merge_all_kernel(int rows_heads, int num_ranks, int num_splits, const float* __restrict__ part_o,
             const float* __restrict__ part_m, const float* __restrict__ part_l,
             __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
             float* __restrict__ rank_lse) {
  const int rh = blockIdx.x;  // row * H + head
  const int n = num_ranks * num_splits;
  const int d = threadIdx.x * 4;
  // one pass with a running maximum M: a batch's m, l and o loads are all in flight
  // together, and the sums are rescaled by 2^(M_old - M_new) when M rises
  float M = -INFINITY;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  for (int i0 = 0; i0 < n; i0 += kBatch) {
    float m[kBatch], l[kBatch];
    float4 o[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      m[u] = -INFINITY;
      l[u] = 0.f;
      o[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i0 + u < n) {  // no load at all past the last partial
        const int64_t idx = (int64_t)(i0 + u) * rows_heads + rh;
        m[u] = part_m[idx];
        l[u] = part_l[idx];
        o[u] = *reinterpret_cast<const float4*>(part_o + idx * kDv + d);
      }
    }
    float Mb = M;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const bool use = i0 + u < n && m[u] != -INFINITY && l[u] > 0.f;
      if (!use) m[u] = -INFINITY;
      Mb = fmaxf(Mb, m[u]);
    }
    if (Mb == -INFINITY) continue;  // nothing so far
    if (Mb != M) {
      const float a = M == -INFINITY ? 0.f : exp2f(M - Mb);
      den *= a;
      acc.x *= a;
      acc.y *= a;
      acc.z *= a;
      acc.w *= a;
      M = Mb;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const float w = m[u] == -INFINITY ? 0.f : exp2f(m[u] - M) * l[u];
      const float4 ov = m[u] == -INFINITY ? make_float4(0.f, 0.f, 0.f, 0.f) : o[u];
      den += w;
      acc.x = fmaf(w, ov.x, acc.x);
      acc.y = fmaf(w, ov.y, acc.y);
      acc.z = fmaf(w, ov.z, acc.z);
      acc.w = fmaf(w, ov.w, acc.w);
    }
  }
  const float inv = den > 0.f ? 1.0f / den : 0.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(out + (int64_t)rh * kDv + d);
  dst[0] = lo;
  dst[1] = hi;
  if (threadIdx.x == 0) lse[rh] = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
  if (rank_lse != nullptr)
    write_rank_lse(rh, rows_heads, num_ranks, num_splits, part_m, part_l, rank_lse, threadIdx.x,
                   blockDim.x);
}

__global__ void __launch_bounds__(32 * kLiveWarps)
merge_live_kernel(int rows_heads, int num_ranks, int num_splits, const float* __restrict__ part_o,
                  const float* __restrict__ part_m, const float* __restrict__ part_l,
                  __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                  float* __restrict__ rank_lse) {
  const int lane = threadIdx.x & 31;
  const int n = num_ranks * num_splits;
  for (int rh = blockIdx.x * kLiveWarps + (threadIdx.x >> 5); rh < rows_heads;
       rh += gridDim.x * kLiveWarps) {
    // one pass with a running maximum M, raised once per 32 partials
    float M = -INFINITY, den = 0.f;
    float acc[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) acc[c] = 0.f;
    for (int c0 = 0; c0 < n; c0 += 32) {
      const int i = c0 + lane;
      float mi = -INFINITY, li = 0.f;
      if (i < n) {
        mi = part_m[(int64_t)i * rows_heads + rh];
        li = part_l[(int64_t)i * rows_heads + rh];
      }
      const bool live = mi != -INFINITY && li > 0.f;
      if (!live) mi = -INFINITY;
      unsigned mask = __ballot_sync(0xffffffffu, live);
      if (mask == 0u) continue;
      float cm = mi;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
      if (cm > M) {
        const float a = M == -INFINITY ? 0.f : exp2f(M - cm);
        den *= a;
#pragma unroll
        for (int c = 0; c < 16; ++c) acc[c] *= a;
        M = cm;
      }
      const float wi = live ? exp2f(mi - M) * li : 0.f;
      while (mask != 0u) {  // warp-uniform: four live partials per round
        int src[4];
        float w[4];
        float4 o[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          src[u] = mask != 0u ? __ffs(mask) - 1 : -1;
          if (mask != 0u) mask &= mask - 1u;
          w[u] = __shfl_sync(0xffffffffu, wi, src[u] < 0 ? 0 : src[u]);
          if (src[u] >= 0) {
            const float4* po = reinterpret_cast<const float4*>(
                part_o + ((int64_t)(c0 + src[u]) * rows_heads + rh) * kDv + 16 * lane);
#pragma unroll
            for (int q = 0; q < 4; ++q) o[u][q] = po[q];
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (src[u] < 0) continue;
          den += w[u];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            acc[4 * q] = fmaf(w[u], o[u][q].x, acc[4 * q]);
            acc[4 * q + 1] = fmaf(w[u], o[u][q].y, acc[4 * q + 1]);
            acc[4 * q + 2] = fmaf(w[u], o[u][q].z, acc[4 * q + 2]);
            acc[4 * q + 3] = fmaf(w[u], o[u][q].w, acc[4 * q + 3]);
          }
        }
      }
    }
    const float inv = den > 0.f ? 1.0f / den : 0.f;
    uint32_t wd[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      __nv_bfloat162 t = __floats2bfloat162_rn(acc[2 * e] * inv, acc[2 * e + 1] * inv);
      wd[e] = *reinterpret_cast<uint32_t*>(&t);
    }
    // 8-byte stores: the interface promises out 8-byte alignment only
    uint2* dst = reinterpret_cast<uint2*>(out + (int64_t)rh * kDv + 16 * lane);
#pragma unroll
    for (int e = 0; e < 4; ++e) dst[e] = make_uint2(wd[2 * e], wd[2 * e + 1]);
    if (lane == 0) lse[rh] = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
    if (rank_lse != nullptr)
      write_rank_lse(rh, rows_heads, num_ranks, num_splits, part_m, part_l, rank_lse, lane, 32);
  }
}

}  // namespace

cudaError_t launch_merge(const dcp_mla_dims& d, const Derived& x, int num_ranks,
                         const float* part_o, const float* part_m, const float* part_l,
                         void* out, float* lse, float* rank_lse, uint32_t* status,
                         cudaStream_t stream) {
  (void)status;
  const int rows_heads = x.rows * d.num_heads;
  if (d.base_splits > 0 && d.base_splits < d.num_splits) {
    const int ctas = std::max(1, std::min((rows_heads + kLiveWarps - 1) / kLiveWarps, 152 * 8));
    merge_live_kernel<<<ctas, 32 * kLiveWarps, 0, stream>>>(
        rows_heads, num_ranks, d.num_splits, part_o, part_m, part_l,
        reinterpret_cast<__nv_bfloat16*>(out), lse, rank_lse);
  } else {
    merge_all_kernel<<<rows_heads, kMergeThreads, 0, stream>>>(
        rows_heads, num_ranks, d.num_splits, part_o, part_m, part_l,
        reinterpret_cast<__nv_bfloat16*>(out), lse, rank_lse);
  }
  return cudaGetLastError();
}

}  // namespace dcpmla
