// Backward pass of scaled dot-product attention on the CUDA cores (fp32
// arithmetic; fp32 or bf16 storage): the gradients dq, dk, dv of a loss
// through softmax(q k^T * scale) v, for training (trishampatil.com,
// "Training (Teacher Forcing + Masking)": the whole target sequence goes
// through one parallel forward pass under the causal mask and the gradients
// flow back through every layer at once).
//
// By the chain rule through the forward's steps, with w_ij the softmax
// weights and dout the incoming gradient:
//   dP_ij = dout_i . v_j                      (through the value sum)
//   D_i   = sum_j w_ij dP_ij = dout_i . out_i
//   dS_ij = w_ij (dP_ij - D_i)                (through the softmax)
//   dq_i  = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i,
//   dv_j  = sum_i w_ij dout_i                 (through the scores)
// Three kernels, no atomics:
//   stats  one warp per query row: lse_i (log2 units, over the allowed keys;
//          +inf for a row with no key or a padded row, so every weight
//          2^(s - lse) of such a row is 0) and D_i
//   dkdv   one warp per 32 keys of a key/value head, a lane per key; the rows
//          of every query head of the group stream through shared memory
//   dq     one warp per 32 query rows, a lane per row; keys and values
//          stream through shared memory
// With the weights recomputed from lse, masked keys are skipped explicitly.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace mha {

namespace {

constexpr int kMaxD = 128;

__device__ __forceinline__ float ldf(const float *p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ldf(const __nv_bfloat16 *p, int64_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void stf(float *p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void stf(__nv_bfloat16 *p, int64_t i, float x) {
  p[i] = __float2bfloat16_rn(x);
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// element offset of (b, head, pos, c) in a tensor of `heads` heads, `len`
// positions and `d` columns, in either layout
__device__ __forceinline__ int64_t at(int layout, int b, int head, int pos, int c, int heads,
                                      int len, int d) {
  if (layout == kLayoutBHSD)
    return ((static_cast<int64_t>(b) * heads + head) * len + pos) * d + c;
  return ((static_cast<int64_t>(b) * len + pos) * heads + head) * d + c;
}

__device__ __forceinline__ int clamp_len(const Problem &p, int b) {
  if (!(p.mask & (kMaskKeyPadding | kMaskQueryPadding))) return p.Lk;
  const int l = p.key_lengths[b];
  return l < 0 ? 0 : (l > p.Lk ? p.Lk : l);
}

// may query row i read key j
__device__ __forceinline__ bool allowed(const Problem &p, int len, int i, int j) {
  if ((p.mask & kMaskQueryPadding) && i >= len) return false;
  if ((p.mask & kMaskCausal) && j > i) return false;
  if ((p.mask & kMaskKeyPadding) && j >= len) return false;
  if ((p.mask & kMaskCausalTail) && j > len - p.Lq + i) return false;
  return true;
}

// ---- stats: lse and D, one warp per query row ------------------------------
template <typename T>
__global__ void __launch_bounds__(128)
    bwd_stats_simt_kernel(const T *__restrict__ q, const T *__restrict__ k,
                          const T *__restrict__ out, const T *__restrict__ dout,
                          float *__restrict__ lse, float *__restrict__ dsum, Problem p) {
  __shared__ float sq[4][kMaxD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + warp;  // (b*H + h)*Lq + i
  const bool live = row < static_cast<int64_t>(p.B) * p.H * p.Lq;
  const int i = live ? static_cast<int>(row % p.Lq) : 0;
  const int bh = live ? static_cast<int>(row / p.Lq) : 0;
  const int b = bh / p.H, h = bh % p.H, hk = h / (p.H / p.Hkv);
  if (live)
    for (int c = lane; c < p.dk; c += 32) sq[warp][c] = ldf(q, at(p.layout, b, h, i, c, p.H, p.Lq, p.dk));
  __syncwarp();
  if (!live) return;
  const int len = clamp_len(p, b);
  float m = -INFINITY, l = 0.f;
  for (int j = lane; j < p.Lk; j += 32) {
    if (!allowed(p, len, i, j)) continue;
    float dot = 0.f;
    for (int c = 0; c < p.dk; ++c)
      dot = fmaf(sq[warp][c], ldf(k, at(p.layout, b, hk, j, c, p.Hkv, p.Lk, p.dk)), dot);
    const float s = dot * p.scale_log2;
    if (s > m) {
      l = l * fast_exp2(m - s) + 1.f;
      m = s;
    } else {
      l += fast_exp2(s - m);
    }
  }
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float L = m == -INFINITY ? 0.f : l * fast_exp2(m - M);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  float dd = 0.f;
  for (int c = lane; c < p.dv; c += 32)
    dd = fmaf(ldf(dout, at(p.layout, b, h, i, c, p.H, p.Lq, p.dv)),
              ldf(out, at(p.layout, b, h, i, c, p.H, p.Lq, p.dv)), dd);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, o);
  if (lane == 0) {
    lse[row] = L > 0.f ? M + log2f(L) : INFINITY;
    dsum[row] = dd;
  }
}

// ---- dk, dv: one warp per 32 keys ------------------------------------------
template <typename T>
__global__ void __launch_bounds__(32)
    bwd_dkdv_simt_kernel(const T *__restrict__ q, const T *__restrict__ k,
                         const T *__restrict__ v, const T *__restrict__ dout,
                         const float *__restrict__ lse, const float *__restrict__ dsum,
                         T *__restrict__ dk, T *__restrict__ dv, Problem p, float scale) {
  extern __shared__ float smem[];
  const int dkk = p.dk, dvv = p.dv;
  float *skr = smem;                   // [32][dk+1] key rows
  float *svr = skr + 32 * (dkk + 1);   // [32][dv+1] value rows
  float *adk = svr + 32 * (dvv + 1);   // [32][dk+1] dk accumulators
  float *adv = adk + 32 * (dkk + 1);   // [32][dv+1] dv accumulators
  float *sq = adv + 32 * (dvv + 1);    // [dk] current query row
  float *sdo = sq + dkk;               // [dv] its incoming gradient
  const int lane = threadIdx.x;
  const int j0 = blockIdx.x * 32, hk = blockIdx.y, b = blockIdx.z;
  const int j = j0 + lane;
  const bool key = j < p.Lk;
  for (int r = 0; r < 32; ++r) {
    const int jj = j0 + r;
    for (int c = lane; c < dkk; c += 32) {
      skr[r * (dkk + 1) + c] = jj < p.Lk ? ldf(k, at(p.layout, b, hk, jj, c, p.Hkv, p.Lk, dkk)) : 0.f;
      adk[r * (dkk + 1) + c] = 0.f;
    }
    for (int c = lane; c < dvv; c += 32) {
      svr[r * (dvv + 1) + c] = jj < p.Lk ? ldf(v, at(p.layout, b, hk, jj, c, p.Hkv, p.Lk, dvv)) : 0.f;
      adv[r * (dvv + 1) + c] = 0.f;
    }
  }
  __syncwarp();
  const int len = clamp_len(p, b);
  const int group = p.H / p.Hkv;
  for (int h = hk * group; h < (hk + 1) * group; ++h) {
    for (int i = 0; i < p.Lq; ++i) {
      const int64_t row = (static_cast<int64_t>(b) * p.H + h) * p.Lq + i;
      for (int c = lane; c < dkk; c += 32) sq[c] = ldf(q, at(p.layout, b, h, i, c, p.H, p.Lq, dkk));
      for (int c = lane; c < dvv; c += 32) sdo[c] = ldf(dout, at(p.layout, b, h, i, c, p.H, p.Lq, dvv));
      __syncwarp();
      if (key && allowed(p, len, i, j)) {
        const float* kr = skr + lane * (dkk + 1);
        const float* vr = svr + lane * (dvv + 1);
        float s = 0.f, dp = 0.f;
        for (int c = 0; c < dkk; ++c) s = fmaf(sq[c], kr[c], s);
        for (int c = 0; c < dvv; ++c) dp = fmaf(sdo[c], vr[c], dp);
        const float w = fast_exp2(s * p.scale_log2 - lse[row]);
        const float ds = w * (dp - dsum[row]);
        float *ak = adk + lane * (dkk + 1);
        float *av = adv + lane * (dvv + 1);
        for (int c = 0; c < dkk; ++c) ak[c] = fmaf(ds, sq[c], ak[c]);
        for (int c = 0; c < dvv; ++c) av[c] = fmaf(w, sdo[c], av[c]);
      }
      __syncwarp();
    }
  }
  for (int r = 0; r < 32; ++r) {
    const int jj = j0 + r;
    if (jj >= p.Lk) break;
    for (int c = lane; c < dkk; c += 32)
      stf(dk, at(p.layout, b, hk, jj, c, p.Hkv, p.Lk, dkk), scale * adk[r * (dkk + 1) + c]);
    for (int c = lane; c < dvv; c += 32)
      stf(dv, at(p.layout, b, hk, jj, c, p.Hkv, p.Lk, dvv), adv[r * (dvv + 1) + c]);
  }
}

// ---- dq: one warp per 32 query rows ----------------------------------------
template <typename T>
__global__ void __launch_bounds__(32)
    bwd_dq_simt_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                       const T *__restrict__ dout, const float *__restrict__ lse,
                       const float *__restrict__ dsum, T *__restrict__ dq, Problem p,
                       float scale) {
  extern __shared__ float smem[];
  const int dkk = p.dk, dvv = p.dv;
  float *sqr = smem;                  // [32][dk+1] query rows
  float *sdo = sqr + 32 * (dkk + 1);  // [32][dv+1] their incoming gradients
  float *adq = sdo + 32 * (dvv + 1);  // [32][dk+1] dq accumulators
  float *sk = adq + 32 * (dkk + 1);   // [dk] current key row
  float *sv = sk + dkk;               // [dv] current value row
  const int lane = threadIdx.x;
  const int i0 = blockIdx.x * 32, h = blockIdx.y, b = blockIdx.z;
  const int hk = h / (p.H / p.Hkv);
  const int i = i0 + lane;
  const bool qrow = i < p.Lq;
  for (int r = 0; r < 32; ++r) {
    const int ii = i0 + r;
    for (int c = lane; c < dkk; c += 32) {
      sqr[r * (dkk + 1) + c] = ii < p.Lq ? ldf(q, at(p.layout, b, h, ii, c, p.H, p.Lq, dkk)) : 0.f;
      adq[r * (dkk + 1) + c] = 0.f;
    }
    for (int c = lane; c < dvv; c += 32)
      sdo[r * (dvv + 1) + c] = ii < p.Lq ? ldf(dout, at(p.layout, b, h, ii, c, p.H, p.Lq, dvv)) : 0.f;
  }
  __syncwarp();
  const int len = clamp_len(p, b);
  const int64_t row = (static_cast<int64_t>(b) * p.H + h) * p.Lq + (qrow ? i : 0);
  const float my_lse = qrow ? lse[row] : INFINITY, my_d = qrow ? dsum[row] : 0.f;
  for (int j = 0; j < p.Lk; ++j) {
    for (int c = lane; c < dkk; c += 32) sk[c] = ldf(k, at(p.layout, b, hk, j, c, p.Hkv, p.Lk, dkk));
    for (int c = lane; c < dvv; c += 32) sv[c] = ldf(v, at(p.layout, b, hk, j, c, p.Hkv, p.Lk, dvv));
    __syncwarp();
    if (qrow && allowed(p, len, i, j)) {
      const float *qr = sqr + lane * (dkk + 1);
      const float *dr = sdo + lane * (dvv + 1);
      float s = 0.f, dp = 0.f;
      for (int c = 0; c < dkk; ++c) s = fmaf(qr[c], sk[c], s);
      for (int c = 0; c < dvv; ++c) dp = fmaf(dr[c], sv[c], dp);
      const float w = fast_exp2(s * p.scale_log2 - my_lse);
      const float ds = w * (dp - my_d);
      float *aq = adq + lane * (dkk + 1);
      for (int c = 0; c < dkk; ++c) aq[c] = fmaf(ds, sk[c], aq[c]);
    }
    __syncwarp();
  }
  for (int r = 0; r < 32; ++r) {
    const int ii = i0 + r;
    if (ii >= p.Lq) break;
    for (int c = lane; c < dkk; c += 32)
      stf(dq, at(p.layout, b, h, ii, c, p.H, p.Lq, dkk), scale * adq[r * (dkk + 1) + c]);
  }
}

template <typename T>
cudaError_t launch_bwd_simt_t(const BwdArgs &a, const Problem &p, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(p.B) * p.H * p.Lq;
  if (rows > 0) {
    const int64_t nblk = (rows + 3) / 4;
    if (nblk > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    bwd_stats_simt_kernel<T><<<static_cast<unsigned>(nblk), 128, 0, stream>>>(
        static_cast<const T *>(a.q), static_cast<const T *>(a.k), static_cast<const T *>(a.out),
        static_cast<const T *>(a.dout), a.lse, a.dsum, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (p.Lk > 0 && p.B > 0 && p.Hkv > 0) {
    const size_t sm = sizeof(float) * (2 * 32 * (p.dk + 1) + 2 * 32 * (p.dv + 1) + p.dk + p.dv);
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(bwd_dkdv_simt_kernel<T>), static_cast<int>(sm));
    if (e != cudaSuccess) return e;
    dim3 grid((p.Lk + 31) / 32, p.Hkv, p.B);
    bwd_dkdv_simt_kernel<T><<<grid, 32, sm, stream>>>(
        static_cast<const T *>(a.q), static_cast<const T *>(a.k), static_cast<const T *>(a.v),
        static_cast<const T *>(a.dout), a.lse, a.dsum, static_cast<T *>(a.dk),
        static_cast<T *>(a.dv), p, a.scale);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (rows > 0) {
    const size_t sm = sizeof(float) * (2 * 32 * (p.dk + 1) + 32 * (p.dv + 1) + p.dk + p.dv);
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(bwd_dq_simt_kernel<T>), static_cast<int>(sm));
    if (e != cudaSuccess) return e;
    dim3 grid((p.Lq + 31) / 32, p.H, p.B);
    bwd_dq_simt_kernel<T><<<grid, 32, sm, stream>>>(
        static_cast<const T *>(a.q), static_cast<const T *>(a.k), static_cast<const T *>(a.v),
        static_cast<const T *>(a.dout), a.lse, a.dsum, static_cast<T *>(a.dq), p, a.scale);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd_simt(const BwdArgs &a, const Problem &p, bool bf16, cudaStream_t stream) {
  if (p.dk > kMaxD || p.dv > kMaxD) return cudaErrorInvalidValue;
  if (p.B > 65535 || p.H > 65535) return cudaErrorInvalidConfiguration;
  return bf16 ? launch_bwd_simt_t<__nv_bfloat16>(a, p, stream)
              : launch_bwd_simt_t<float>(a, p, stream);
}

}  // namespace mha
