// The step after the path: the cross-rank exchange in the all-to-all wire format.
//
// "Context Parallel Guide (PCP & DCP)", Decode and comm_backend "a2a": every rank
// returns its output and LSE; ONE all-to-all carries each rank's output with the
// LSE packed alongside it, and the destination combines locally, so that every
// rank ends with its slice of the heads. The fp32 LSE travels as two 16-bit
// halves of the BF16 buffer (bit for bit); the output travels as BF16.
//
// Wire format of the chunk a source rank sends to destination d (which owns heads
// [d*Hg, (d+1)*Hg), Hg = H / dcp): [R][Hg][P] BF16 outputs, then [R][Hg][2] LSE
// halves (low 16 bits, then high 16 bits of the float32), then zero words up to a
// multiple of 8 words. A source's send buffer is [dcp][chunk].
//
//   a2a_pack_kernel     one warp per (rank, row, head), grid-stride: merges the
//                       rank's splits (m, l, o) into its normalised output, RNE to
//                       BF16, and its natural-log LSE, written into the chunk for
//                       the head's destination. HBM-bound: reads NS*(2 KiB + 8 B),
//                       writes 1 KiB + 4 B per (rank, row, head).
//   a2a_combine_kernel  one warp per (destination, row, head of its slice): reads
//                       the dcp source entries, LSE-weights them. HBM-bound: reads
//                       dcp*(2P + 4) B, writes 2P + 4 B per (row, head).
//
// Project-before-merge ("enable_project_before_merge" on the same page): each
// rank's BF16 output is projected by the head's W_V before it is sent, so P = the
// projected width instead of 512.
//
//   a2a_project_kernel  one CTA per (head, 128 vectors), a vector being one (rank,
//                       row) entry of packed send buffers: D[128][P] =
//                       A[128][512] . W_V[h]^T on the tensor cores (tcgen05, M = 128,
//                       N = P, K = 512 in 8 chunks of 64, fp32 accumulator in tensor
//                       memory). The threads copy the chunk's A rows and W_V rows
//                       into 128-byte-swizzled K-major tiles with coalesced loads
//                       (the next chunk's loads are in flight meanwhile). Two
//                       stages: the stores of chunk c overlap the MMAs of chunk c-1. The epilogue reads D back (tcgen05.ld), rounds to
//                       BF16 and writes the projected entries; the LSE words are
//                       copied.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "sm103.cuh"

namespace dcpmla {
namespace {

using namespace sm103;

constexpr float kLn2 = 0.6931471805599453f;

constexpr int kXWarps = 8;  // warps (entries in flight) per CTA of pack and combine

// 8 floats, each times scale, as 8 BF16 values (one 16-byte chunk)
__device__ __forceinline__ uint4 f32_to_bf16x8(const float (&f)[8], float scale) {
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    __nv_bfloat162 t = __floats2bfloat162_rn(f[2 * e] * scale, f[2 * e + 1] * scale);
    w[e] = *reinterpret_cast<uint32_t*>(&t);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// One warp per (rank, row, head) entry, grid-stride: lane l owns dims [16l, 16l + 16).
// More than one split: one pass with a running maximum, the sums rescaled by
// 2^(M_old - M_new) when M rises; kPackAll reads four splits' m, l and outputs
// together (every slot expected to hold work), kPackLive reads the m and l of 32
// splits first and then only the live splits' outputs (wave balancing leaves most
// slots empty; a skipped slot's m is -inf). One split (kPackOne): its normalised
// output as it is and LSE = (m + log2 l) ln 2 (the same arithmetic as the partial
// kernel's packed epilogue, so both give the same bits).
enum { kPackOne = 0, kPackAll = 1, kPackLive = 2 };
template <int kMode>
__global__ void __launch_bounds__(32 * kXWarps, kMode == kPackOne ? 4 : 2)
a2a_pack_kernel(int R, int H, int G, int num_splits, int num_ranks, int64_t cw,
                const float* __restrict__ part_o, const float* __restrict__ part_m,
                const float* __restrict__ part_l, uint16_t* __restrict__ send) {
  const int rows_heads = R * H;
  const int Hg = H / G;
  const int lane = threadIdx.x & 31;
  const int64_t n_entries = (int64_t)num_ranks * rows_heads;
  const int64_t stride = (int64_t)gridDim.x * kXWarps;
  for (int64_t e = (int64_t)blockIdx.x * kXWarps + (threadIdx.x >> 5); e < n_entries;
       e += stride) {
    const int k = (int)(e / rows_heads);
    const int rh = (int)(e - (int64_t)k * rows_heads);
    const int row = rh / H, h = rh - row * H;
    const int d = h / Hg, hl = h - d * Hg;
    const int64_t p0 = (int64_t)k * num_splits * rows_heads + rh;  // split 0 of this rank
    uint16_t* chunk = send + ((int64_t)k * G + d) * cw;
    if (rh == 0) {  // the zero words that end each of this rank's chunks
      const int64_t used = (int64_t)R * Hg * (kDv + 2);
      for (int dd = 0; dd < G; ++dd)
        for (int64_t w = used + lane; w < cw; w += 32) send[((int64_t)k * G + dd) * cw + w] = 0;
    }
    float M = -INFINITY, den = 0.f;
    float acc[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) acc[c] = 0.f;
    float lse;
    if (kMode == kPackOne) {
      // the output's loads do not wait for m and l: a dead entry's values are dropped
      const float4* src = reinterpret_cast<const float4*>(part_o + p0 * kDv + 16 * lane);
      float4 v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] = src[q];
      const float m = part_m[p0], l = part_l[p0];
      const bool live = m != -INFINITY && l > 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[4 * q] = live ? v[q].x : 0.f;
        acc[4 * q + 1] = live ? v[q].y : 0.f;
        acc[4 * q + 2] = live ? v[q].z : 0.f;
        acc[4 * q + 3] = live ? v[q].w : 0.f;
      }
      den = live ? 1.f : 0.f;
      lse = live ? (m + log2f(l)) * kLn2 : -INFINITY;
    } else {
      if (kMode == kPackAll) {
        for (int s0 = 0; s0 < num_splits; s0 += 4) {
          float m[4], l[4];
          float4 o[4][4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            m[u] = -INFINITY;
            l[u] = 0.f;
            if (s0 + u < num_splits) {  // no load at all past the last split
              const int64_t i = p0 + (int64_t)(s0 + u) * rows_heads;
              m[u] = part_m[i];
              l[u] = part_l[i];
              const float4* src = reinterpret_cast<const float4*>(part_o + i * kDv + 16 * lane);
#pragma unroll
              for (int q = 0; q < 4; ++q) o[u][q] = src[q];
            } else {
#pragma unroll
              for (int q = 0; q < 4; ++q) o[u][q] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
          float Mb = M;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (!(m[u] != -INFINITY && l[u] > 0.f)) m[u] = -INFINITY;
            Mb = fmaxf(Mb, m[u]);
          }
          if (Mb == -INFINITY) continue;
          if (Mb != M) {
            const float a = M == -INFINITY ? 0.f : exp2f(M - Mb);
            den *= a;
#pragma unroll
            for (int c = 0; c < 16; ++c) acc[c] *= a;
            M = Mb;
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (m[u] == -INFINITY) continue;
            const float w = exp2f(m[u] - M) * l[u];
            den += w;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              acc[4 * q] = fmaf(w, o[u][q].x, acc[4 * q]);
              acc[4 * q + 1] = fmaf(w, o[u][q].y, acc[4 * q + 1]);
              acc[4 * q + 2] = fmaf(w, o[u][q].z, acc[4 * q + 2]);
              acc[4 * q + 3] = fmaf(w, o[u][q].w, acc[4 * q + 3]);
            }
          }
        }
      } else {
        // m and l of 32 splits in one load per lane; only live splits' outputs are read,
        // four at a time (an empty split, or a slot the partial kernel skipped, is -inf)
        for (int c0 = 0; c0 < num_splits; c0 += 32) {
          float mi = -INFINITY, li = 0.f;
          if (c0 + lane < num_splits) {
            mi = part_m[p0 + (int64_t)(c0 + lane) * rows_heads];
            li = part_l[p0 + (int64_t)(c0 + lane) * rows_heads];
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
          while (mask != 0u) {  // warp-uniform
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
                    part_o + (p0 + (int64_t)(c0 + src[u]) * rows_heads) * kDv + 16 * lane);
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
      }
      lse = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
    }
    const float inv =
        kMode == kPackOne ? (den > 0.f ? 1.f : 0.f) : (den > 0.f ? 1.0f / den : 0.f);
    float lo[8], hi[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) lo[c] = acc[c], hi[c] = acc[8 + c];
    uint4* dst = reinterpret_cast<uint4*>(chunk + ((int64_t)row * Hg + hl) * kDv + 16 * lane);
    dst[0] = f32_to_bf16x8(lo, inv);
    dst[1] = f32_to_bf16x8(hi, inv);
    if (lane == 0) {
      uint32_t* lp = reinterpret_cast<uint32_t*>(chunk + (int64_t)R * Hg * kDv +
                                                 ((int64_t)row * Hg + hl) * 2);
      *lp = __float_as_uint(lse);  // the low 16 bits first, then the high (little-endian)
    }
  }
}

// kW BF16 values (kW = 4: 8 bytes, kW = 8: 16 bytes) as one load or store
template <int kW> struct BfVec;
template <> struct BfVec<4> {
  using T = uint2;
  static __device__ __forceinline__ void words(const T& v, uint32_t (&w)[2]) { w[0] = v.x, w[1] = v.y; }
  static __device__ __forceinline__ T make(const uint32_t (&w)[2]) { return make_uint2(w[0], w[1]); }
};
template <> struct BfVec<8> {
  using T = uint4;
  static __device__ __forceinline__ void words(const T& v, uint32_t (&w)[4]) {
    w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
  }
  static __device__ __forceinline__ T make(const uint32_t (&w)[4]) {
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// Lanes given to one combine entry of nch chunks: the power of two at or above nch, at
// most 32.
__host__ __device__ inline int lanes_per_entry(int nch) {
  int l = 1;
  while (l < nch && l < 32) l <<= 1;
  return l;
}

// One warp per (destination, row, head of its slice), grid-stride: lane l owns the
// kW-value chunks l, l + 32, ... of the P values (narrow payloads: lpe lanes per
// entry, several entries per warp). One pass over the sources with a
// running maximum of their LSEs (natural log), four sources' loads in flight together.
template <int kW>
__global__ void __launch_bounds__(32 * kXWarps)
a2a_combine_kernel(int R, int H, int G, int P, int num_dst, const uint16_t* __restrict__ recv,
                   int64_t src_stride, int64_t dst_stride, int dst_begin,
                   __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  using V = BfVec<kW>;
  using T = typename V::T;
  constexpr int kC = kDv / kW / 32;  // chunks per lane at the largest payload
  constexpr int kSrc = 4;            // sources whose loads are in flight together
  const int Hg = H / G;
  const int nch = P / kW;
  // a warp combines 32 / lpe entries side by side (no lane talks to another)
  const int lpe = lanes_per_entry(nch);
  const int epw = 32 / lpe;
  const int lane = (threadIdx.x & 31) & (lpe - 1);
  const int64_t per_dst = (int64_t)R * Hg;
  const int64_t n_entries = (int64_t)num_dst * per_dst;
  const int64_t stride = (int64_t)gridDim.x * kXWarps * epw;
  for (int64_t g = ((int64_t)blockIdx.x * kXWarps + (threadIdx.x >> 5)) * epw +
                   (threadIdx.x & 31) / lpe;
       g < n_entries; g += stride) {
    const int di = (int)(g / per_dst);
    const int e = (int)(g - (int64_t)di * per_dst);  // row * Hg + hl
    const int row = e / Hg, hl = e - row * Hg;
    const int h = (dst_begin + di) * Hg + hl;
    const uint16_t* base = recv + (int64_t)di * dst_stride;
    const int64_t lse_off = (int64_t)R * Hg * P + (int64_t)e * 2;
    float M = -INFINITY, den = 0.f;
    float acc[kC][kW];
#pragma unroll
    for (int c = 0; c < kC; ++c)
#pragma unroll
      for (int q = 0; q < kW; ++q) acc[c][q] = 0.f;
    for (int s0 = 0; s0 < G; s0 += kSrc) {
      float ls[kSrc];
      T v[kSrc][kC];
#pragma unroll
      for (int u = 0; u < kSrc; ++u) {
        const int s = s0 + u;
        ls[u] = -INFINITY;
        if (s < G) {
          const uint16_t* src = base + (int64_t)s * src_stride;
          ls[u] = __uint_as_float(*reinterpret_cast<const uint32_t*>(src + lse_off));
          const T* ent = reinterpret_cast<const T*>(src + (int64_t)e * P);
#pragma unroll
          for (int c = 0; c < kC; ++c)
            if (lane + lpe * c < nch) v[u][c] = ent[lane + lpe * c];
        }
      }
      float Mb = M;
#pragma unroll
      for (int u = 0; u < kSrc; ++u) Mb = fmaxf(Mb, ls[u]);
      if (Mb == -INFINITY) continue;
      if (Mb != M) {
        const float a = M == -INFINITY ? 0.f : expf(M - Mb);
        den *= a;
#pragma unroll
        for (int c = 0; c < kC; ++c)
#pragma unroll
          for (int q = 0; q < kW; ++q) acc[c][q] *= a;
        M = Mb;
      }
#pragma unroll
      for (int u = 0; u < kSrc; ++u) {
        if (ls[u] == -INFINITY) continue;
        const float w = expf(ls[u] - M);
        den += w;
#pragma unroll
        for (int c = 0; c < kC; ++c) {
          if (lane + lpe * c >= nch) continue;
          uint32_t wd[kW / 2];
          V::words(v[u][c], wd);
#pragma unroll
          for (int q = 0; q < kW / 2; ++q) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wd[q]));
            acc[c][2 * q] = fmaf(w, f.x, acc[c][2 * q]);
            acc[c][2 * q + 1] = fmaf(w, f.y, acc[c][2 * q + 1]);
          }
        }
      }
    }
    const float inv = den > 0.f ? 1.0f / den : 0.f;
    T* dst = reinterpret_cast<T*>(out + ((int64_t)row * H + h) * P);
#pragma unroll
    for (int c = 0; c < kC; ++c) {
      if (lane + lpe * c >= nch) continue;
      uint32_t wd[kW / 2];
#pragma unroll
      for (int q = 0; q < kW / 2; ++q) {
        __nv_bfloat162 t = __floats2bfloat162_rn(acc[c][2 * q] * inv, acc[c][2 * q + 1] * inv);
        wd[q] = *reinterpret_cast<uint32_t*>(&t);
      }
      dst[lane + lpe * c] = V::make(wd);
    }
    if (lane == 0) lse[(int64_t)row * H + h] = den > 0.f ? M + logf(den) : -INFINITY;
  }
}

// Grid of a warp-per-entry kernel: every entry covered, at most a few waves of the
// SMs' resident CTAs (the loop strides over the rest).
static unsigned entry_grid(int64_t n_entries) {
  const int64_t want = (n_entries + kXWarps - 1) / kXWarps;
  return (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, 152 * 8));
}

constexpr int kProjVecs = 128;                  // vectors per CTA (MMA M)
constexpr int kProjChunk = 64;                  // K dims per stage (one 128-byte swizzle atom)
constexpr int kProjABytes = kProjVecs * 128;    // A tile of one chunk
constexpr uint32_t kProjTmemCols = 256;         // accumulator, P <= 256
constexpr int kProjMinSmem = 80 * 1024;         // at most two CTAs (2 x 256 columns) per SM
constexpr uint64_t kProjTimeoutNs = 4000000000ull;

__device__ bool proj_wait(uint64_t* bar, uint32_t parity, uint32_t* status) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_wait_sleep(a, parity)) {
    if (globaltimer_ns() - t0 > kProjTimeoutNs) {
      raise_status(status, DCP_STATUS_TIMEOUT);
      return false;
    }
  }
  return true;
}

__global__ void __launch_bounds__(128)
a2a_project_kernel(int R, int H, int G, int num_ranks, int P, int64_t cw_in, int64_t cw,
                   const uint16_t* __restrict__ send_in, const uint16_t* __restrict__ w_v,
                   uint16_t* __restrict__ send, uint32_t* status) {
  extern __shared__ unsigned char smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int stage_bytes = kProjABytes + P * 128;  // multiple of 1024 (P % 16 == 0)
  // bars[0..1]: the MMAs of a stage completed; bars[2]: drain after a timeout
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + 2 * stage_bytes);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  const int tid = threadIdx.x;
  const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
  const int h = blockIdx.x;
  const int Hg = H / G, d = h / Hg, hl = h % Hg;
  const int v = blockIdx.y * kProjVecs + tid;  // this thread's vector = A row = TMEM lane
  const bool valid = v < num_ranks * R;
  const int k = valid ? v / R : 0, row = valid ? v % R : 0;
  const int64_t entry = (int64_t)row * Hg + hl;
  const uint16_t* in_chunk = send_in + ((int64_t)k * G + d) * cw_in;

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_init(&bars[2], 1);
    *abort_flag = 0;
    fence_mbarrier_init_cluster();
  }
  if (warp == 0) {
    tmem_alloc(tslot, kProjTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = __shfl_sync(0xffffffffu, *tslot, 0);
  const uint32_t idesc = idesc_f16(kProjVecs, P, true, false);
  const uint32_t sbase = smem_u32(base);
  // Loads are coalesced: in every chunk, thread tid moves 16-byte piece j = tid % 8 of
  // A rows 16i + tid / 8 (i = 0..7) and of W_V rows 16i + tid / 8 (i < P / 16), so a
  // warp reads four whole 128-byte row segments per instruction. One chunk ahead.
  const int jp = tid & 7, r0 = tid >> 3;
  const uint4* asrc[8];  // this thread's A rows (nullptr: past the last vector)
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int vi = blockIdx.y * kProjVecs + 16 * i + r0;
    asrc[i] = nullptr;
    if (vi < num_ranks * R) {
      const int ki = vi / R, ri = vi - ki * R;
      asrc[i] = reinterpret_cast<const uint4*>(send_in + ((int64_t)ki * G + d) * cw_in +
                                               ((int64_t)ri * Hg + hl) * kDv) + jp;
    }
  }
  const uint4* wsrc = reinterpret_cast<const uint4*>(w_v + ((int64_t)h * P + r0) * kDv) + jp;
  const int nb = P / 16;  // W_V rows per thread
  uint4 cur[8], bcur[16];
  auto fetch = [&](int c) {
#pragma unroll
    for (int i = 0; i < 8; ++i) cur[i] = asrc[i] ? asrc[i][c * 8] : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (i < nb) bcur[i] = wsrc[(int64_t)16 * i * (kDv / 8) + c * 8];
  };
  fetch(0);

  for (int c = 0; c < kDv / kProjChunk; ++c) {
    const int st = c & 1;
    uint8_t* A = base + st * stage_bytes;
    uint8_t* B = A + kProjABytes;
    // the MMAs of chunk c-2 read this stage: one thread waits (bounded), and nobody
    // writes the stage unless that wait succeeded
    if (c >= 2) {
      if (tid == 0 && !proj_wait(&bars[st], ((c - 2) >> 1) & 1, status)) *abort_flag = 1;
      __syncthreads();
      if (*abort_flag) break;
    }
    // row r of a tile: the chunk's 8 groups of 8 dims, group j at 16-byte slot j ^ (r & 7)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = 16 * i + r0;
      *reinterpret_cast<uint4*>(A + r * 128 + ((jp ^ (r & 7)) << 4)) = cur[i];
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int r = 16 * i + r0;
      if (i < nb) *reinterpret_cast<uint4*>(B + r * 128 + ((jp ^ (r & 7)) << 4)) = bcur[i];
    }
    if (c + 1 < kDv / kProjChunk) fetch(c + 1);
    fence_proxy_async_smem();  // the tensor core reads the tiles (async proxy)
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
      tc_fence_after();
      if (elect_one()) {
        const uint32_t a_addr = sbase + st * stage_bytes;
        const uint32_t b_addr = a_addr + kProjABytes;
#pragma unroll
        for (int kk = 0; kk < kProjChunk / 16; ++kk)
          mma_f16_ss(tbase, smem_desc_sw128(a_addr + kk * 32, 16, 1024),
                     smem_desc_sw128(b_addr + kk * 32, 16, 1024), idesc,
                     (c > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&bars[st]);
      }
      __syncwarp();
    }
  }
  // chunks 6 and 7 were the fourth commits of their barriers (phase 3); after a
  // timeout, every MMA issued so far is drained instead before TMEM is read or freed
  if (tid == 0 && !*abort_flag &&
      !(proj_wait(&bars[0], 1, status) && proj_wait(&bars[1], 1, status)))
    *abort_flag = 1;
  __syncthreads();
  const bool aborted = *abort_flag != 0;
  if (aborted) {
    if (warp == 0) tc_commit_elect(&bars[2]);
    if (tid == 0) proj_wait(&bars[2], 0, status);
    __syncthreads();
  }
  tc_fence_after();

  uint16_t* chunk = send + ((int64_t)k * G + d) * cw;
  const uint32_t trow = tbase + ((uint32_t)(warp * 32) << 16);
  for (int c16 = 0; c16 < (aborted ? 0 : P / 16); ++c16) {
    uint32_t r[16];
    tmem_ld16(trow + 16 * c16, r);
    tmem_wait_ld16(r);
    if (valid) {
      uint32_t wd[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(r[2 * q]),
                                                  __uint_as_float(r[2 * q + 1]));
        wd[q] = *reinterpret_cast<uint32_t*>(&b2);
      }
      uint4* dst = reinterpret_cast<uint4*>(chunk + entry * P + 16 * c16);
      dst[0] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
      dst[1] = make_uint4(wd[4], wd[5], wd[6], wd[7]);
    }
  }
  if (valid && !aborted) {
    const uint16_t* lin = in_chunk + (int64_t)R * Hg * kDv + entry * 2;
    uint16_t* lp = chunk + (int64_t)R * Hg * P + entry * 2;
    lp[0] = lin[0];
    lp[1] = lin[1];
  }
  if (blockIdx.x == 0 && blockIdx.y == 0) {  // the zero words that end every chunk
    const int64_t used = (int64_t)R * Hg * (P + 2);
    for (int kd = 0; kd < num_ranks * G; ++kd)
      for (int64_t w = used + tid; w < cw; w += blockDim.x) send[(int64_t)kd * cw + w] = 0;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, kProjTmemCols);
  }
}

}  // namespace

int64_t a2a_chunk_words(int R, int Hg, int P) {
  const int64_t lse_words = 2 * (int64_t)R * Hg;
  return (int64_t)R * Hg * P + (lse_words + 7) / 8 * 8;
}

cudaError_t launch_a2a_pack(const dcp_mla_dims& d, const Derived& x, int num_ranks,
                            const float* part_o, const float* part_m, const float* part_l,
                            void* send, cudaStream_t stream) {
  const int G = d.dcp;
  const int64_t cw = a2a_chunk_words(x.rows, d.num_heads / G, kDv);
  const int64_t n = (int64_t)num_ranks * x.rows * d.num_heads;
  auto kern = d.num_splits == 1                                     ? a2a_pack_kernel<kPackOne>
              : d.base_splits > 0 && d.base_splits < d.num_splits ? a2a_pack_kernel<kPackLive>
                                                                   : a2a_pack_kernel<kPackAll>;
  kern<<<entry_grid(n), 32 * kXWarps, 0, stream>>>(
      x.rows, d.num_heads, G, d.num_splits, num_ranks, cw, part_o, part_m, part_l,
      reinterpret_cast<uint16_t*>(send));
  return cudaGetLastError();
}

cudaError_t launch_a2a_project(const dcp_mla_dims& d, const Derived& x, int num_ranks,
                               const void* send_in, const void* w_v, int payload, void* send,
                               uint32_t* status, cudaStream_t stream) {
  const int G = d.dcp;
  const int64_t cw_in = a2a_chunk_words(x.rows, d.num_heads / G, kDv);
  const int64_t cw = a2a_chunk_words(x.rows, d.num_heads / G, payload);
  const int smem = max(1024 + 2 * (kProjABytes + payload * 128) + 64, kProjMinSmem);
  static int attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (attr_set[dev] < smem) {
    e = cudaFuncSetAttribute(a2a_project_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = smem;
  }
  const int64_t vecs = (int64_t)num_ranks * x.rows;
  dim3 grid((unsigned)d.num_heads, (unsigned)((vecs + kProjVecs - 1) / kProjVecs));
  a2a_project_kernel<<<grid, 128, smem, stream>>>(
      x.rows, d.num_heads, G, num_ranks, payload, cw_in, cw,
      reinterpret_cast<const uint16_t*>(send_in), reinterpret_cast<const uint16_t*>(w_v),
      reinterpret_cast<uint16_t*>(send), status);
  return cudaGetLastError();
}

cudaError_t launch_a2a_combine(const dcp_mla_dims& d, const Derived& x, int payload,
                               const void* recv, int64_t src_stride, int64_t dst_stride,
                               int dst_begin, int num_dst, void* out, float* lse,
                               cudaStream_t stream) {
  const int G = d.dcp;
  const int64_t n = (int64_t)num_dst * x.rows * (d.num_heads / G);
  // 16-byte chunks when every entry and the output rows start on a 16-byte boundary
  const bool wide = payload % 8 == 0 && ((uintptr_t)out & 15) == 0;
  const int nch = payload / (wide ? 8 : 4);
  const int lpe = lanes_per_entry(nch);
  auto kern = wide ? a2a_combine_kernel<8> : a2a_combine_kernel<4>;
  kern<<<entry_grid((n + 32 / lpe - 1) / (32 / lpe)), 32 * kXWarps, 0, stream>>>(
      x.rows, d.num_heads, G, payload, num_dst, reinterpret_cast<const uint16_t*>(recv),
      src_stride, dst_stride, dst_begin, reinterpret_cast<__nv_bfloat16*>(out), lse);
  return cudaGetLastError();
}

}  // namespace dcpmla
