// fp32 scaled dot-product attention on the CUDA cores (FFMA only, no TF32).
//
// One CTA = one (batch, head) and 16 query rows (with shared key/value heads,
// query head h reads head h / (H / H_kv); either tensor layout); each of its 4 warps owns 4
// rows.  Keys/values stream through shared memory 32 at a time (one key per
// lane); each row keeps a running max and running sum (online softmax) so the
// n x n score matrix is never stored.  Steps follow the four of "Scaled
// Dot-Product Attention: Step by Step": lane j forms q_i . k_j (step 1), the
// scale is folded with log2(e) (step 2), exp2 against the running max with
// warp-shuffle reductions (step 3), and the weighted sum of value rows
// (step 4) accumulates in fp32 with each lane owning d_v/32 output columns.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace mha {

namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;  // 16
constexpr int kKeysPerTile = 32;
constexpr int kMaxD = 128;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Element offset of row 0 of one head, and the stride between its rows, in a
// contiguous tensor of `heads` heads, `len` rows and `d` columns.
struct HeadView {
  int64_t base, row;
};
__device__ __forceinline__ HeadView head_view(int layout, int b, int head, int heads, int len,
                                              int d) {
  if (layout == kLayoutBHSD)
    return {(static_cast<int64_t>(b) * heads + head) * len * d, static_cast<int64_t>(d)};
  return {(static_cast<int64_t>(b) * len * heads + head) * d, static_cast<int64_t>(heads) * d};
}

__global__ void __launch_bounds__(kWarps * 32)
    attn_f32_simt_kernel(const float *__restrict__ q, const float *__restrict__ k,
                         const float *__restrict__ v, float *__restrict__ out, Problem p) {
  extern __shared__ float smem[];
  const int dk = p.dk, dv = p.dv;
  const int ks = dk + 1;  // padded key-row stride: lanes read different rows conflict-free
  float *sq = smem;                                 // [16][dk]
  float *sk = sq + kRowsPerCta * dk;                // [32][dk+1]
  float *sv = sk + kKeysPerTile * ks;               // [32][dv]

  const int n_qblk = (p.Lq + kRowsPerCta - 1) / kRowsPerCta;
  const int64_t bh = blockIdx.x / n_qblk;
  const int q0 = (blockIdx.x % n_qblk) * kRowsPerCta;
  const int b = static_cast<int>(bh / p.H), h = static_cast<int>(bh % p.H);
  const int hkv = h / (p.H / p.Hkv);  // key/value head this query head reads
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int len = p.Lk;
  if (p.mask & (kMaskKeyPadding | kMaskQueryPadding)) {
    int l = p.key_lengths[b];
    len = l < 0 ? 0 : (l > p.Lk ? p.Lk : l);
  }
  int kv_end = p.Lk;
  if (p.mask & kMaskKeyPadding) kv_end = len;
  if (p.mask & kMaskCausal) kv_end = min(kv_end, min(q0 + kRowsPerCta, p.Lq));
  // cached decoding: the block's last query sits at position len - Lq + its row
  if (p.mask & kMaskCausalTail)
    kv_end = max(min(kv_end, len - p.Lq + min(q0 + kRowsPerCta, p.Lq)), 0);

  const HeadView vq = head_view(p.layout, b, h, p.H, p.Lq, dk);
  const HeadView vk = head_view(p.layout, b, hkv, p.Hkv, p.Lk, dk);
  const HeadView vv = head_view(p.layout, b, hkv, p.Hkv, p.Lk, dv);
  const HeadView vo = head_view(p.layout, b, h, p.H, p.Lq, dv);
  const float *qb = q + vq.base;
  const float *kb = k + vk.base;
  const float *vb = v + vv.base;
  float *ob = out + vo.base;

  for (int e = threadIdx.x; e < kRowsPerCta * dk; e += blockDim.x) {
    const int r = e / dk, c = e % dk;
    sq[e] = (q0 + r < p.Lq) ? qb[(q0 + r) * vq.row + c] : 0.f;
  }

  float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][kMaxD / 32];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int t = 0; t < kMaxD / 32; ++t) acc[r][t] = 0.f;
  }

  for (int kv0 = 0; kv0 < kv_end; kv0 += kKeysPerTile) {
    __syncthreads();  // previous tile fully consumed (and sq written, first time)
    for (int e = threadIdx.x; e < kKeysPerTile * dk; e += blockDim.x) {
      const int j = e / dk, c = e % dk;
      sk[j * ks + c] = (kv0 + j < p.Lk) ? kb[(kv0 + j) * vk.row + c] : 0.f;
    }
    for (int e = threadIdx.x; e < kKeysPerTile * dv; e += blockDim.x) {
      const int j = e / dv, c = e % dv;
      sv[e] = (kv0 + j < p.Lk) ? vb[(kv0 + j) * vv.row + c] : 0.f;
    }
    __syncthreads();

    const int j = kv0 + lane;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int lr = warp * kRowsPerWarp + r;
      const int i = q0 + lr;
      // step 1: q_i . k_j
      float dot = 0.f;
      const float *qr = sq + lr * dk;
      const float *kr = sk + lane * ks;
      for (int c = 0; c < dk; ++c) dot = fmaf(qr[c], kr[c], dot);
      bool ok = (j < kv_end) && (i < p.Lq);
      if (p.mask & kMaskCausal) ok = ok && (j <= i);
      if (p.mask & kMaskCausalTail) ok = ok && (j <= len - p.Lq + i);
      // step 2 (scale, in log2 units) and step 3 (online softmax)
      const float x = ok ? dot * p.scale_log2 : -INFINITY;
      const float m_new = fmaxf(m[r], warp_max(x));
      if (m_new == -INFINITY) continue;  // nothing allowed yet in this row
      const float alpha = fast_exp2(m[r] - m_new);
      const float pj = fast_exp2(x - m_new);
      l[r] = l[r] * alpha + warp_sum(pj);
      m[r] = m_new;
      // step 4: weighted sum of value rows
#pragma unroll
      for (int t = 0; t < kMaxD / 32; ++t) acc[r][t] *= alpha;
      for (int jj = 0; jj < kKeysPerTile; ++jj) {
        const float pw = __shfl_sync(0xffffffffu, pj, jj);
#pragma unroll
        for (int t = 0; t < kMaxD / 32; ++t) {
          const int c = lane + 32 * t;
          if (c < dv) acc[r][t] = fmaf(pw, sv[jj * dv + c], acc[r][t]);
        }
      }
    }
  }

#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int i = q0 + warp * kRowsPerWarp + r;
    if (i >= p.Lq) continue;
    const bool zero_row = (l[r] == 0.f) || ((p.mask & kMaskQueryPadding) && i >= len);
    const float inv = zero_row ? 0.f : 1.f / l[r];
    if (p.lse != nullptr && lane == 0)
      p.lse[(static_cast<size_t>(b) * p.H + h) * p.Lq + i] =
          zero_row ? INFINITY : m[r] + __log2f(l[r]);
#pragma unroll
    for (int t = 0; t < kMaxD / 32; ++t) {
      const int c = lane + 32 * t;
      if (c < dv) ob[i * vo.row + c] = zero_row ? 0.f : acc[r][t] * inv;
    }
  }
}

__global__ void zero_fill_kernel(uint4 *__restrict__ out, size_t n16, uint8_t *__restrict__ tail,
                                 size_t ntail) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16; i += stride)
    out[i] = make_uint4(0, 0, 0, 0);
  if (blockIdx.x == 0)
    for (size_t i = threadIdx.x; i < ntail; i += blockDim.x) tail[i] = 0;
}

}  // namespace

cudaError_t launch_f32_simt(const float *q, const float *k, const float *v, float *out,
                            const Problem &p, cudaStream_t stream) {
  const int n_qblk = (p.Lq + kRowsPerCta - 1) / kRowsPerCta;
  const int64_t grid = static_cast<int64_t>(p.B) * p.H * n_qblk;
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  const size_t smem =
      sizeof(float) * (kRowsPerCta * p.dk + kKeysPerTile * (p.dk + 1) + kKeysPerTile * p.dv);
  if (smem > 48 * 1024) {
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(attn_f32_simt_kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  attn_f32_simt_kernel<<<static_cast<unsigned>(grid), kWarps * 32, smem, stream>>>(q, k, v, out,
                                                                                  p);
  return cudaGetLastError();
}

__global__ void fill_f32_kernel(float *__restrict__ dst, size_t n, float value) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n; i += stride)
    dst[i] = value;
}

cudaError_t launch_fill_f32(float *dst, size_t n, float value, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  unsigned grid = static_cast<unsigned>(n / 256 + 1);
  if (grid > 4096) grid = 4096;
  fill_f32_kernel<<<grid, 256, 0, stream>>>(dst, n, value);
  return cudaGetLastError();
}

cudaError_t launch_zero_fill(void *out, size_t bytes, cudaStream_t stream) {
  const size_t n16 = bytes / 16;
  const size_t ntail = bytes - n16 * 16;
  unsigned grid = static_cast<unsigned>(n16 / 256 + 1);
  if (grid > 4096) grid = 4096;
  zero_fill_kernel<<<grid, 256, 0, stream>>>(static_cast<uint4 *>(out), n16,
                                             static_cast<uint8_t *>(out) + n16 * 16, ntail);
  return cudaGetLastError();
}

}  // namespace mha
