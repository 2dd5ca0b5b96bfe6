// Step 4: LSE merge of every split of every rank into the BF16 output.
//
// "Context Parallel Guide (PCP & DCP)", Decode: the per-rank partial outputs
// are LSE-corrected and summed. "[ROCm][MLA][DCP] Support causal multi-token
// verification", Implementation item 3: base-2 partial statistics become a BF16
// output plus a natural-log LSE. Splits and ranks are merged in one pass: with
// m, l, o per (rank, split), M = max m, w = 2^(m - M) * l,
// O = sum w*o / sum w, LSE = (M + log2 sum w) * ln 2 (M kept as a running maximum).
//
// HBM-bound: one CTA per (row, head) reads nr*NS partial rows of 512 floats with
// 16-byte coalesced loads and writes 1 KB of BF16.
#include <cuda_bf16.h>

#include "common.cuh"

namespace dcpmla {
namespace {

constexpr int kMergeThreads = 128;  // 4 dims per thread
constexpr int kBatch = 4;           // partials whose loads are issued together
constexpr float kLn2 = 0.6931471805599453f;

__global__ void __launch_bounds__(kMergeThreads)
merge_kernel(int rows_heads, int num_ranks, int num_splits, const float* __restrict__ part_o,
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
  if (rank_lse != nullptr) {
    for (int k = threadIdx.x; k < num_ranks; k += blockDim.x) {
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
}

}  // namespace

cudaError_t launch_merge(const dcp_mla_dims& d, const Derived& x, int num_ranks,
                         const float* part_o, const float* part_m, const float* part_l,
                         void* out, float* lse, float* rank_lse, uint32_t* status,
                         cudaStream_t stream) {
  (void)status;
  const int rows_heads = x.rows * d.num_heads;
  merge_kernel<<<rows_heads, kMergeThreads, 0, stream>>>(
      rows_heads, num_ranks, d.num_splits, part_o, part_m, part_l,
      reinterpret_cast<__nv_bfloat16*>(out), lse, rank_lse);
  return cudaGetLastError();
}

}  // namespace dcpmla
