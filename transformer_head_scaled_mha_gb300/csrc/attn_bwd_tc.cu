// Backward pass of scaled dot-product attention on the tcgen05 tensor cores
// (bf16, d in {64, 128}): the gradients dq, dk, dv of a loss through
// softmax(q k^T * scale) v, for training (trishampatil.com, "Training (Teacher
// Forcing + Masking)": the whole target sequence goes through one parallel
// forward pass under the causal mask and the gradients flow back through
// every layer at once).  By the chain rule through the forward's steps, with
// w_ij the softmax weights and dout the incoming gradient:
//
//   dP = dout V^T,  D_i = dout_i . out_i,  dS = w * (dP - D)  (row-wise D)
//   dq = scale dS K,  dk = scale dS^T Q,  dv = w^T dout
//
// Three kernels, no atomics, every product on the tensor cores with fp32
// accumulators in TMEM; the weights are recomputed from the per-row
// log-sum-exp (log2 units), w_ij = 2^(s_ij * scale * log2(e) - lse_i):
//
//   stats  per 128 query rows: S = Q K^T tile by tile, the running max and
//          sum (moved lazily, as in the forward), lse; D from out and dout
//          (+inf lse for a row that attends to nothing: all its weights 0)
//   dq     per 128 query rows: S = Q K_j^T and dP = dout V_j^T, then the
//          softmax warpgroup (thread = row) forms dS (bf16) over S_j in
//          TMEM, and dQ += dS K_j reads it from TMEM as the A operand.  S is
//          double-buffered, so S_{j+1} overlaps the softmax of tile j, and
//          dP_{j+1} goes ahead of dQ_j
//   dkdv   per 128 keys of a key/value head, over the query tiles of every
//          query head of the group, 64 queries at a time: S^T = K Q^T and
//          dP^T = V dout^T (keys on the lanes), then thread = key forms w^T
//          and dS^T (bf16) over them in TMEM, and dV += w^T dout,
//          dK += dS^T Q read them as A operands; two score buffers let one
//          half's softmax overlap the other half's products, w^T forms while
//          dP^T is computed, and dV starts before dS^T is ready
//
// Warp roles (192 threads): warps 0-3 softmax (thread r = TMEM lane r),
// warp 4 TMA producer, warp 5 TMEM owner and MMA issuer.  Operand tiles are
// [128 rows x 64] 128B-swizzled blocks written by TMA; the row-major K, V,
// Q and dout tiles serve as K-major operands of the score products and as
// MN-major B operands of the gradient products.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kThreads = 192;
constexpr int kWg = 128;   // softmax threads
constexpr int kT = 128;    // rows of every tile (queries or keys)
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kMaxSlots = 8;
constexpr int kBand = 8;  // tiles per band of the CTA order

// CTA order of the per-tile kernels: bands of kBand tiles, heaviest band
// first; inside a band, a head's tiles side by side.  The CTAs running at one
// time then cover few heads, and those that read a head's other operand tiles
// read the same ones at about the same time, mostly from L2.  Tile i of `n`
// (0 = heaviest) and head index of CTA x over `heads` heads.
__device__ __forceinline__ void band_order(int x, int heads, int n, int &head, int &i) {
  const int full = n / kBand;  // full bands; a partial one (the lightest) ends the order
  const int t = min(x / (heads * kBand), full);
  const int lo = t * kBand;
  const int size = min(kBand, n - lo);
  const int local = x - t * heads * kBand;
  head = local / size;
  i = lo + local % size;
}

template <int D>
struct Geo {
  static constexpr int kBlk = 128 * 128;             // one [128 x 64] swizzle block
  static constexpr int kTile = (D / 64) * kBlk;      // one [128 x D] tile
};

__device__ __forceinline__ int clamp_len(const Problem &p, int b) {
  if (!(p.mask & (kMaskKeyPadding | kMaskQueryPadding))) return p.Lk;
  const int l = p.key_lengths[b];
  return l < 0 ? 0 : (l > p.Lk ? p.Lk : l);
}

// keys j < row_limit(i) may be read by query row i (0: none)
__device__ __forceinline__ int row_limit(const Problem &p, int len, int i) {
  if ((p.mask & kMaskQueryPadding) && i >= len) return 0;
  int jmax = p.Lk;
  if (p.mask & kMaskKeyPadding) jmax = min(jmax, len);
  if (p.mask & kMaskCausal) jmax = min(jmax, i + 1);
  if (p.mask & kMaskCausalTail) jmax = max(min(jmax, len - p.Lq + i + 1), 0);
  return jmax;
}

// key tiles [0, n) that the query rows [q0, q0 + 128) of one head can read
__device__ __forceinline__ int key_tiles(const Problem &p, int len, int q0) {
  if ((p.mask & kMaskQueryPadding) && q0 >= len) return 0;
  const int q1 = min(q0 + kT, p.Lq);  // one past the tile's last row
  int kv_end = p.Lk;
  if (p.mask & kMaskKeyPadding) kv_end = min(kv_end, len);
  if (p.mask & kMaskCausal) kv_end = min(kv_end, q1);
  if (p.mask & kMaskCausalTail) kv_end = min(kv_end, len - p.Lq + q1);
  return kv_end > 0 ? (kv_end + kT - 1) / kT : 0;
}

// element offset of row (b, head, pos) in a tensor of `heads` heads, `len`
// positions and d columns
__device__ __forceinline__ size_t row_at(int layout, int b, int head, int pos, int heads, int len,
                                         int d) {
  const size_t r = layout == kLayoutBHSD ? (static_cast<size_t>(b) * heads + head) * len + pos
                                         : (static_cast<size_t>(b) * len + pos) * heads + head;
  return r * d;
}

// 32 fp32 values * f -> bf16, 64 bytes at dst (16-byte aligned)
__device__ __forceinline__ void store_row32(uint16_t *dst, const uint32_t (&v)[32], float f) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    w.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]) * f, __uint_as_float(v[8 * q + 1]) * f);
    w.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]) * f, __uint_as_float(v[8 * q + 3]) * f);
    w.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]) * f, __uint_as_float(v[8 * q + 5]) * f);
    w.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]) * f, __uint_as_float(v[8 * q + 7]) * f);
    st_global_v4(dst + 8 * q, w);
  }
}
__device__ __forceinline__ void store_zero32(uint16_t *dst) {
#pragma unroll
  for (int q = 0; q < 4; ++q) st_global_v4(dst + 8 * q, make_uint4(0u, 0u, 0u, 0u));
}

// D/16 steps of a [128 x D] x [128 x D]^T product, both operands K-major
template <int D>
__device__ __forceinline__ void mma_scores(uint32_t d_tmem, uint32_t sa, uint32_t sb,
                                           uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk >> 2) * Geo<D>::kBlk + (kk & 3) * 32;
    tc_mma_ss(d_tmem, smem_desc_sw128(sa + off, 16, 1024), smem_desc_sw128(sb + off, 16, 1024),
              idesc, kk > 0 ? 1u : 0u);
  }
}
// 8 steps of A[128 x 128 bf16 in TMEM] x B[128 rows x D, MN-major smem]
template <int D>
__device__ __forceinline__ void mma_grad(uint32_t d_tmem, uint32_t a_tmem, uint32_t sb,
                                         uint32_t idesc, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < kT / 16; ++kk)
    tc_mma_ts(d_tmem, a_tmem + kk * 8, smem_desc_sw128(sb + kk * 16 * 128, Geo<D>::kBlk, 1024),
              idesc, (accumulate || kk > 0) ? 1u : 0u);
}

// ============================================================================
// stats: lse and D per query row
// ============================================================================
// two CTAs per SM (256 TMEM columns and under half the shared memory each):
// one CTA's softmax runs while the tensor core serves the other
template <int D>
struct StatsCfg {
  static constexpr int kSlots = D == 128 ? 2 : 4;
  static constexpr size_t kSmem = 1024 + static_cast<size_t>(1 + kSlots) * Geo<D>::kTile + 512;
};
struct StatsBars {
  uint64_t q_full;
  uint64_t k_full[kMaxSlots], k_empty[kMaxSlots];
  uint64_t s_full[2], s_free[2];
  uint32_t tmem_base;
  int abort_flag;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    bwd_stats_tc_kernel(const __grid_constant__ LongMaps maps, const Problem p, const BwdArgs a) {
  using C = StatsCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *q_smem = smem;
  uint8_t *k_smem = q_smem + Geo<D>::kTile;
  StatsBars *bars = reinterpret_cast<StatsBars *>(k_smem + C::kSlots * Geo<D>::kTile);
  volatile int *abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BH = p.B * p.H;
  const int nqb = (p.Lq + kT - 1) / kT;
  int bh, qi;
  band_order(static_cast<int>(blockIdx.x), BH, nqb, bh, qi);
  const int q0 = (nqb - 1 - qi) * kT;  // heaviest (causal) first
  const int b = bh / p.H, h = bh % p.H, hk = h / (p.H / p.Hkv);
  const int len = clamp_len(p, b);
  const int nt = key_tiles(p, len, q0);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], kWg);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars->tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  int issued = 0;
  uint64_t *last_commit = nullptr;
  uint32_t last_parity = 0;

  if (warp == 4) {
    if (lane == 0 && nt > 0) {
      mbar_arrive_expect_tx(&bars->q_full, Geo<D>::kTile);
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_4d(q_smem + blk * Geo<D>::kBlk, &maps.q, &bars->q_full, blk * 64, q0, h, b);
      for (int j = 0; j < nt; ++j) {
        const int s = j % C::kSlots, r = j / C::kSlots;
        if (!mbar_wait(&bars->k_empty[s], (r & 1) ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(&bars->k_full[s], Geo<D>::kTile);
        for (int blk = 0; blk < D / 64; ++blk)
          tma_load_4d(k_smem + s * Geo<D>::kTile + blk * Geo<D>::kBlk, &maps.k, &bars->k_full[s],
                      blk * 64, j * kT, hk, b);
        issued = j + 1;
      }
    }
  } else if (warp == 5) {
    const uint32_t idesc = idesc_bf16_f32(128, kT, 0);
    bool ok = nt == 0 || mbar_wait(&bars->q_full, 0, abort_flag);
    for (int j = 0; ok && j < nt; ++j) {
      const int s = j % C::kSlots, r = j / C::kSlots;
      if (!(ok = mbar_wait(&bars->k_full[s], r & 1, abort_flag))) break;
      // S buffer j % 2 held S_{j-2}: the softmax has read it
      if (j >= 2 && !(ok = mbar_wait(&bars->s_free[j & 1], ((j - 2) >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      if (lane == 0) {
        mma_scores<D>(tmem + (j & 1) * kT, smem_addr(q_smem),
                      smem_addr(k_smem + s * Geo<D>::kTile), idesc);
        tc_commit(&bars->s_full[j & 1]);
        tc_commit(&bars->k_empty[s]);
      }
      __syncwarp();
      last_commit = &bars->k_empty[s];
      last_parity = r & 1;
    }
  } else {
    const int r = threadIdx.x;  // tile row = TMEM lane
    const int i = q0 + r;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int jmax = i < p.Lq ? row_limit(p, len, i) : 0;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[j & 1], (j >> 1) & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) tmem_ld32(tmem + lane_base + (j & 1) * kT + ch * 32, sr[ch]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars->s_free[j & 1]);
      const int lim = min(max(jmax - j * kT, 0), kT);
      const bool need_mask = __any_sync(0xffffffffu, lim < kT);
      // positive scale: max over the raw scores, then one FMA per score (the
      // same rounding as the weights the gradient kernels form)
      const bool pos = p.scale_log2 > 0.f;
      const float mt = pos ? mask_max128(sr, need_mask, 0, lim) * p.scale_log2
                           : scale_mask_max128(sr, p.scale_log2, need_mask, 0, lim);
      if (mt > m + kRescaleThreshold) {
        if (m != -INFINITY) l *= ex2_approx(m - mt);
        m = mt;
      }
      l += pos ? exp2_fma_sum128(sr, p.scale_log2, m, m != -INFINITY)
               : exp2_sum128(sr, m, m != -INFINITY);
    }
    if (ok && i < p.Lq) {
      const size_t row = (static_cast<size_t>(b) * p.H + h) * p.Lq + i;
      a.lse[row] = l > 0.f ? m + __log2f(l) : INFINITY;
      const uint16_t *o = static_cast<const uint16_t *>(a.out) +
                          row_at(p.layout, b, h, i, p.H, p.Lq, D);
      const uint16_t *g = static_cast<const uint16_t *>(a.dout) +
                          row_at(p.layout, b, h, i, p.H, p.Lq, D);
      float dsum = 0.f;
#pragma unroll 4
      for (int c = 0; c < D; c += 8) {
        const uint4 ov = *reinterpret_cast<const uint4 *>(o + c);
        const uint4 gv = *reinterpret_cast<const uint4 *>(g + c);
        const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          dsum = fmaf(__uint_as_float(ow[t] << 16), __uint_as_float(gw[t] << 16), dsum);
          dsum = fmaf(__uint_as_float(ow[t] & 0xffff0000u), __uint_as_float(gw[t] & 0xffff0000u),
                      dsum);
        }
      }
      a.dsum[row] = dsum;
    }
  }

  if (*abort_flag && warp == 4 && lane == 0) {
    for (int idx = issued - C::kSlots; idx < issued; ++idx)
      if (idx >= 0) (void)wait_teardown(&bars->k_full[idx % C::kSlots], (idx / C::kSlots) & 1);
    if (nt > 0) (void)wait_teardown(&bars->q_full, 0);
  }
  if (*abort_flag && warp == 5 && lane == 0 && last_commit != nullptr)
    (void)wait_teardown(last_commit, last_parity);
  if (*abort_flag && threadIdx.x == 0) atomicExch(p.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, 256);
}

// dS = w (dP - D) over 32 key columns for the calling thread's row: sv, pv the
// row's S and dP, columns c < lim allowed (others weight 0), lse and D the
// row's.  A chunk the whole warp may read takes packed fp32 pairs, no mask.
__device__ __forceinline__ void dq_chunk(const uint32_t (&sv)[32], const uint32_t (&pv)[32],
                                         int lim, float scale_log2, float lse, float dd,
                                         uint32_t (&pk)[16]) {
  if (__all_sync(0xffffffffu, lim >= 32)) {
    const uint64_t sc = f2_pack(scale_log2, scale_log2), nl = f2_pack(-lse, -lse);
    const uint64_t d2 = f2_pack(dd, dd);
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      float x0, x1, g0, g1;
      f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sc, nl),
                x0, x1);
      const float w0 = ex2_approx(x0), w1 = ex2_approx(x1);
      f2_unpack(f2_mul(f2_pack(w0, w1),
                       f2_sub(f2_pack(__uint_as_float(pv[e]), __uint_as_float(pv[e + 1])), d2)),
                g0, g1);
      pk[e >> 1] = pack_bf16x2(g0, g1);
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    const float w0 = e < lim ? ex2_approx(__uint_as_float(sv[e]) * scale_log2 - lse) : 0.f;
    const float w1 = e + 1 < lim ? ex2_approx(__uint_as_float(sv[e + 1]) * scale_log2 - lse) : 0.f;
    pk[e >> 1] = pack_bf16x2(w0 * (__uint_as_float(pv[e]) - dd),
                             w1 * (__uint_as_float(pv[e + 1]) - dd));
  }
}

// ============================================================================
// dq: per 128 query rows, over the key tiles
// ============================================================================
template <int D>
struct DqCfg {
  // separate K and V rings: K_j is read until dQ_j, V_j only until dP_j, so a
  // third K slot lets K_{j+2} load while dQ_j still holds K_j
  static constexpr int kKSlots = D == 128 ? 3 : 4;
  static constexpr int kVSlots = D == 128 ? 2 : 4;
  static constexpr size_t kSmem =
      1024 + static_cast<size_t>(2 + kKSlots + kVSlots) * Geo<D>::kTile + 512;
  // TMEM: S0, S1 (dS_j bf16 over the first 64 columns of S_j), dP, dQ
  static constexpr uint32_t kS = 0, kDp = 256, kDq = 384;
};
struct DqBars {
  uint64_t qdo_full;
  uint64_t k_full[kMaxSlots], k_empty[kMaxSlots];
  uint64_t v_full[kMaxSlots], v_empty[kMaxSlots];
  uint64_t sdp_full;  // S_j and dP_j in TMEM
  uint64_t ds_full;   // dS_j in TMEM (softmax threads)
  uint64_t dq_done;
  uint32_t tmem_base;
  int abort_flag;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_tc_kernel(const __grid_constant__ LongMaps maps, const Problem p, const BwdArgs a) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *q_smem = smem;                           // Q tile
  uint8_t *do_smem = q_smem + Geo<D>::kTile;        // dout tile
  uint8_t *k_smem = do_smem + Geo<D>::kTile;        // kKSlots K tiles
  uint8_t *v_smem = k_smem + C::kKSlots * Geo<D>::kTile;  // kVSlots V tiles
  DqBars *bars = reinterpret_cast<DqBars *>(v_smem + C::kVSlots * Geo<D>::kTile);
  volatile int *abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BH = p.B * p.H;
  const int nqb = (p.Lq + kT - 1) / kT;
  int bh, qi;
  band_order(static_cast<int>(blockIdx.x), BH, nqb, bh, qi);
  const int qt = nqb - 1 - qi;  // heaviest (causal) first
  const int q0 = qt * kT;
  const int b = bh / p.H, h = bh % p.H, hk = h / (p.H / p.Hkv);
  const int len = clamp_len(p, b);
  const int nt = key_tiles(p, len, q0);

  if (threadIdx.x == 0) {
    mbar_init(&bars->qdo_full, 1);
    for (int s = 0; s < C::kKSlots; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < C::kVSlots; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    mbar_init(&bars->sdp_full, 1);
    mbar_init(&bars->ds_full, kWg);
    mbar_init(&bars->dq_done, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  int k_issued = 0, v_issued = 0;
  uint64_t *last_commit = nullptr;
  uint32_t last_parity = 0;

  if (warp == 4) {
    if (lane == 0 && nt > 0) {
      mbar_arrive_expect_tx(&bars->qdo_full, 2 * Geo<D>::kTile);
      for (int blk = 0; blk < D / 64; ++blk) {
        tma_load_4d(q_smem + blk * Geo<D>::kBlk, &maps.q, &bars->qdo_full, blk * 64, q0, h, b);
        tma_load_4d(do_smem + blk * Geo<D>::kBlk, &maps.o, &bars->qdo_full, blk * 64, q0, h, b);
      }
      for (int j = 0; j < nt; ++j) {
        const int sk = j % C::kKSlots, rk = j / C::kKSlots;
        const int sv = j % C::kVSlots, rv = j / C::kVSlots;
        if (!mbar_wait(&bars->k_empty[sk], (rk & 1) ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(&bars->k_full[sk], Geo<D>::kTile);
        for (int blk = 0; blk < D / 64; ++blk)
          tma_load_4d(k_smem + sk * Geo<D>::kTile + blk * Geo<D>::kBlk, &maps.k, &bars->k_full[sk],
                      blk * 64, j * kT, hk, b);
        k_issued = j + 1;
        if (!mbar_wait(&bars->v_empty[sv], (rv & 1) ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(&bars->v_full[sv], Geo<D>::kTile);
        for (int blk = 0; blk < D / 64; ++blk)
          tma_load_4d(v_smem + sv * Geo<D>::kTile + blk * Geo<D>::kBlk, &maps.v, &bars->v_full[sv],
                      blk * 64, j * kT, hk, b);
        v_issued = j + 1;
      }
    }
  } else if (warp == 5) {
    // S_0, dP_0, S_1; then per tile j, once dS_j is in TMEM: dP_{j+1} (dP_j
    // is in the softmax's registers), dQ_j, and S_{j+2} over S_j (after dQ_j
    // read dS_j: the products of one thread run in issue order)
    const uint32_t idesc_s = idesc_bf16_f32(128, kT, 0);
    const uint32_t idesc_g = idesc_bf16_f32(128, D, 1);
    const uint32_t sq = smem_addr(q_smem), sdo = smem_addr(do_smem);
    auto k_tile = [&](int j) { return smem_addr(k_smem + (j % C::kKSlots) * Geo<D>::kTile); };
    auto v_tile = [&](int j) { return smem_addr(v_smem + (j % C::kVSlots) * Geo<D>::kTile); };
    auto wait_k = [&](int j) {
      return mbar_wait(&bars->k_full[j % C::kKSlots], (j / C::kKSlots) & 1, abort_flag);
    };
    auto wait_v = [&](int j) {
      return mbar_wait(&bars->v_full[j % C::kVSlots], (j / C::kVSlots) & 1, abort_flag);
    };
    bool ok = nt == 0 || (mbar_wait(&bars->qdo_full, 0, abort_flag) && wait_k(0) && wait_v(0));
    if (ok && nt > 0) {
      tc_fence_after();
      if (lane == 0) {
        mma_scores<D>(tmem + C::kS, sq, k_tile(0), idesc_s);
        mma_scores<D>(tmem + C::kDp, sdo, v_tile(0), idesc_s);
        tc_commit(&bars->sdp_full);
        tc_commit(&bars->v_empty[0]);
      }
      __syncwarp();
      if (nt > 1 && (ok = wait_k(1))) {
        tc_fence_after();
        if (lane == 0) mma_scores<D>(tmem + C::kS + kT, sq, k_tile(1), idesc_s);
        __syncwarp();
      }
    }
    for (int j = 0; ok && j < nt; ++j) {
      if (!(ok = mbar_wait(&bars->ds_full, j & 1, abort_flag))) break;
      if (j + 1 < nt && !(ok = wait_v(j + 1))) break;
      tc_fence_after();
      if (lane == 0) {
        if (j + 1 < nt) {
          mma_scores<D>(tmem + C::kDp, sdo, v_tile(j + 1), idesc_s);
          tc_commit(&bars->sdp_full);
          tc_commit(&bars->v_empty[(j + 1) % C::kVSlots]);
        }
        mma_grad<D>(tmem + C::kDq, tmem + C::kS + (j & 1) * kT, k_tile(j), idesc_g, j > 0);
        tc_commit(&bars->k_empty[j % C::kKSlots]);
      }
      __syncwarp();
      last_commit = &bars->k_empty[j % C::kKSlots];
      last_parity = (j / C::kKSlots) & 1;
      if (j + 2 < nt) {
        if (!(ok = wait_k(j + 2))) break;
        tc_fence_after();
        if (lane == 0) mma_scores<D>(tmem + C::kS + (j & 1) * kT, sq, k_tile(j + 2), idesc_s);
        __syncwarp();
      }
    }
    if (ok && nt > 0 && lane == 0) tc_commit(&bars->dq_done);
    __syncwarp();
  } else {
    const int r = threadIdx.x;
    const int i = q0 + r;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const bool row = i < p.Lq;
    const size_t ridx = (static_cast<size_t>(b) * p.H + h) * p.Lq + (row ? i : 0);
    const float lse = row ? a.lse[ridx] : INFINITY;
    const float dd = row ? a.dsum[ridx] : 0.f;
    const int jmax = row ? row_limit(p, len, i) : 0;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->sdp_full, j & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_t = tmem + lane_base + C::kS + (j & 1) * kT;
      const uint32_t dp_t = tmem + lane_base + C::kDp;
      // two chunks of S and dP load from TMEM at once (one wait per pair);
      // the packed dS of chunks 0, 1 lands on S columns [0, 32), which the
      // loads of chunks 2, 3 do not read
      uint32_t sv[2][32], pv[2][32];
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        tmem_ld32(s_t + (2 * c2) * 32, sv[0]);
        tmem_ld32(s_t + (2 * c2 + 1) * 32, sv[1]);
        tmem_ld32(dp_t + (2 * c2) * 32, pv[0]);
        tmem_ld32(dp_t + (2 * c2 + 1) * 32, pv[1]);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int ch = 2 * c2 + cc;
          uint32_t pk[16];
          const int lim = jmax - (j * kT + ch * 32);  // columns c < lim are allowed
          dq_chunk(sv[cc], pv[cc], lim, p.scale_log2, lse, dd, pk);
          tmem_st16(s_t + ch * 16, pk);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->ds_full);
    }
    // the TMEM loads are warp-collective: every thread of the warp takes
    // them; only rows inside the tensor are stored
    if (nt > 0 && ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->dq_done, 0, abort_flag));
      tc_fence_after();
    }
    uint16_t *dst = static_cast<uint16_t *>(a.dq) + (row ? row_at(p.layout, b, h, i, p.H, p.Lq, D) : 0);
#pragma unroll 1
    for (int ch = 0; ok && ch < D / 32; ++ch) {
      if (nt > 0) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + C::kDq + ch * 32, v);
        tmem_wait_ld();
        if (row) store_row32(dst + ch * 32, v, a.scale);
      } else if (row) {
        store_zero32(dst + ch * 32);
      }
    }
  }

  if (*abort_flag && warp == 4 && lane == 0) {
    for (int idx = k_issued - C::kKSlots; idx < k_issued; ++idx)
      if (idx >= 0) (void)wait_teardown(&bars->k_full[idx % C::kKSlots], (idx / C::kKSlots) & 1);
    for (int idx = v_issued - C::kVSlots; idx < v_issued; ++idx)
      if (idx >= 0) (void)wait_teardown(&bars->v_full[idx % C::kVSlots], (idx / C::kVSlots) & 1);
    if (nt > 0) (void)wait_teardown(&bars->qdo_full, 0);
  }
  if (*abort_flag && warp == 5 && lane == 0 && last_commit != nullptr)
    (void)wait_teardown(last_commit, last_parity);
  if (*abort_flag && threadIdx.x == 0) atomicExch(p.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, 512);
}

// ============================================================================
// dkdv: per 128 keys of a key/value head, over its query heads' row tiles
// ============================================================================
template <int D>
struct DkdvCfg {
  static constexpr int kSlots = D == 128 ? 2 : 4;  // ring of (Q tile, dout tile) pairs
  static constexpr int kStat = 2 * kT * 4;          // -lse and D of one query tile
  static constexpr size_t kSmem = 1024 + static_cast<size_t>(2 + 2 * kSlots) * Geo<D>::kTile +
                                  static_cast<size_t>(kSlots) * kStat + 512;
  // TMEM, per 64-query half h of a query tile: S^T_h at 64 h (w^T bf16 over
  // it), dP^T_h at 128 + 64 h (dS^T bf16 over it); then dV, dK
  static constexpr uint32_t kS = 0, kDp = 128, kDv = 256, kDk = 256 + D;
};
struct DkdvBars {
  uint64_t kv_full;
  uint64_t qd_full[kMaxSlots], qd_empty[kMaxSlots];
  uint64_t s_full[2];    // S^T_h in TMEM
  uint64_t dp_full[2];   // dP^T_h in TMEM
  uint64_t w_full[2];    // w^T_h in TMEM (softmax threads)
  uint64_t ds_full[2];   // dS^T_h in TMEM (softmax threads)
  uint64_t pd_free[2];   // dV, dK products of half h done reading them
  uint64_t done;
  uint32_t tmem_base;
  int abort_flag;
};
constexpr int kDkdvThreads = 224;

// w^T over 32 query columns for the calling thread's key: sv its S^T row,
// st the columns' negated lse, columns lo <= e < hi allowed (others weight
// 0); w in fp32 (for dS) and packed bf16 pairs (the dV operand).  A chunk
// the whole warp may read takes packed fp32 pairs and no mask.
__device__ __forceinline__ void dkdv_w32(const uint32_t (&sv)[32], const float *st, int lo,
                                         int hi, float scale_log2, float (&w)[32],
                                         uint32_t (&pw)[16]) {
  if (__all_sync(0xffffffffu, lo <= 0 && hi >= 32)) {
    const uint64_t sc = f2_pack(scale_log2, scale_log2);
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      const float4 l4 = *reinterpret_cast<const float4 *>(st + e);
      float x0, x1, x2, x3;
      f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sc,
                       f2_pack(l4.x, l4.y)),
                x0, x1);
      f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3])), sc,
                       f2_pack(l4.z, l4.w)),
                x2, x3);
      w[e] = ex2_approx(x0);
      w[e + 1] = ex2_approx(x1);
      w[e + 2] = ex2_approx(x2);
      w[e + 3] = ex2_approx(x3);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      const float4 l4 = *reinterpret_cast<const float4 *>(st + e);
      const float l[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
      for (int t = 0; t < 4; ++t)
        w[e + t] = e + t >= lo && e + t < hi
                       ? ex2_approx(fmaf(__uint_as_float(sv[e + t]), scale_log2, l[t]))
                       : 0.f;
    }
  }
#pragma unroll
  for (int e = 0; e < 32; e += 2) pw[e >> 1] = pack_bf16x2(w[e], w[e + 1]);
}

// dS^T = w^T (dP^T - D) over the same 32 columns, packed bf16 pairs (the dK
// operand); st the columns' negated lse, their D kT floats further on
__device__ __forceinline__ void dkdv_ds32(const float (&w)[32], const uint32_t (&pv)[32],
                                          const float *st, uint32_t (&pd)[16]) {
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    const float4 d4 = *reinterpret_cast<const float4 *>(st + kT + e);
    float g0, g1, g2, g3;
    f2_unpack(f2_mul(f2_pack(w[e], w[e + 1]),
                     f2_sub(f2_pack(__uint_as_float(pv[e]), __uint_as_float(pv[e + 1])),
                            f2_pack(d4.x, d4.y))),
              g0, g1);
    f2_unpack(f2_mul(f2_pack(w[e + 2], w[e + 3]),
                     f2_sub(f2_pack(__uint_as_float(pv[e + 2]), __uint_as_float(pv[e + 3])),
                            f2_pack(d4.z, d4.w))),
              g2, g3);
    pd[e >> 1] = pack_bf16x2(g0, g1);
    pd[(e >> 1) + 1] = pack_bf16x2(g2, g3);
  }
}

// query tiles [t_lo, t_hi) that can read some key of [k0, k0 + 128)
__device__ __forceinline__ void query_tiles(const Problem &p, int len, int k0, int &t_lo,
                                            int &t_hi) {
  const int nqb = (p.Lq + kT - 1) / kT;
  t_lo = 0;
  t_hi = nqb;
  if ((p.mask & kMaskKeyPadding) && k0 >= len) t_hi = 0;
  if (p.mask & kMaskQueryPadding) t_hi = min(t_hi, (len + kT - 1) / kT);
  if (p.mask & kMaskCausal) t_lo = max(t_lo, k0 / kT);
  if (p.mask & kMaskCausalTail) t_lo = max(t_lo, max(k0 - len + p.Lq, 0) / kT);
  if (t_lo > t_hi) t_lo = t_hi;
}

// Each query tile is taken as two 64-query halves (N = 64 score products), so
// that with dV and dK holding 2 x D TMEM columns two score buffers still fit:
// the softmax of one half runs while the tensor core computes the other
// half's scores or the previous half's gradients.  Two warps issue -- the
// score products S^T_h = K Q_h^T, dP^T_h = V dout_h^T (warp 5) and the
// gradient products dV += w^T_h dout_h, dK += dS^T_h Q_h (warp 6) -- so that
// the smaller products do not serialise on one issuing thread.
template <int D>
__global__ void __launch_bounds__(kDkdvThreads, 1)
    bwd_dkdv_tc_kernel(const __grid_constant__ LongMaps maps, const Problem p, const BwdArgs a) {
  using C = DkdvCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *k_smem = smem;                        // K tile
  uint8_t *v_smem = k_smem + Geo<D>::kTile;      // V tile
  uint8_t *qd_smem = v_smem + Geo<D>::kTile;     // kSlots x (Q tile, dout tile)
  float *stat = reinterpret_cast<float *>(qd_smem + 2 * C::kSlots * Geo<D>::kTile);  // -lse, D
  DkdvBars *bars = reinterpret_cast<DkdvBars *>(reinterpret_cast<uint8_t *>(stat) +
                                                C::kSlots * C::kStat);
  volatile int *abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BK = p.B * p.Hkv;
  const int nkb = (p.Lk + kT - 1) / kT;
  int bk, kt;
  band_order(static_cast<int>(blockIdx.x), BK, nkb, bk, kt);  // heaviest (causal) first
  const int k0 = kt * kT;
  const int b = bk / p.Hkv, hk = bk % p.Hkv;
  const int group = p.H / p.Hkv;
  const int len = clamp_len(p, b);
  int t_lo, t_hi;
  query_tiles(p, len, k0, t_lo, t_hi);
  const int per_head = t_hi - t_lo;
  const int nw = group * per_head;  // work items (query head of the group, query tile)

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(&bars->qd_full[s], 1);
      mbar_init(&bars->qd_empty[s], 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&bars->s_full[h], 1);
      mbar_init(&bars->dp_full[h], 1);
      mbar_init(&bars->w_full[h], kWg);
      mbar_init(&bars->ds_full[h], kWg);
      mbar_init(&bars->pd_free[h], 1);
    }
    mbar_init(&bars->done, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  int issued = 0;
  uint64_t *last_commit = nullptr;
  uint32_t last_parity = 0;

  if (warp == 4) {
    if (nw > 0) {
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->kv_full, 2 * Geo<D>::kTile);
        for (int blk = 0; blk < D / 64; ++blk) {
          tma_load_4d(k_smem + blk * Geo<D>::kBlk, &maps.k, &bars->kv_full, blk * 64, k0, hk, b);
          tma_load_4d(v_smem + blk * Geo<D>::kBlk, &maps.v, &bars->kv_full, blk * 64, k0, hk, b);
        }
      }
      for (int w = 0; w < nw; ++w) {
        const int s = w % C::kSlots, r = w / C::kSlots;
        const int h = hk * group + w / per_head, q0 = (t_lo + w % per_head) * kT;
        // the tile's -lse and D (rows past Lq: weight 0), all in flight at once
        // and before the slot is free, so that their latency hides in the wait
        const size_t row0 = (static_cast<size_t>(b) * p.H + h) * p.Lq;
        float lse_r[kT / 32], dsum_r[kT / 32];
#pragma unroll
        for (int i = 0; i < kT / 32; ++i) {
          const int e = lane + 32 * i;
          const bool in = q0 + e < p.Lq;
          lse_r[i] = in ? -a.lse[row0 + q0 + e] : -INFINITY;  // negated
          dsum_r[i] = in ? a.dsum[row0 + q0 + e] : 0.f;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->qd_empty[s], (r & 1) ^ 1, abort_flag)))
          break;
        float *st = stat + s * (C::kStat / 4);
#pragma unroll
        for (int i = 0; i < kT / 32; ++i) {
          st[lane + 32 * i] = lse_r[i];
          st[kT + lane + 32 * i] = dsum_r[i];
        }
        __syncwarp();
        if (lane == 0) {
          uint8_t *dst = qd_smem + 2 * s * Geo<D>::kTile;
          mbar_arrive_expect_tx(&bars->qd_full[s], 2 * Geo<D>::kTile);
          for (int blk = 0; blk < D / 64; ++blk) {
            tma_load_4d(dst + blk * Geo<D>::kBlk, &maps.q, &bars->qd_full[s], blk * 64, q0, h, b);
            tma_load_4d(dst + Geo<D>::kTile + blk * Geo<D>::kBlk, &maps.o, &bars->qd_full[s],
                        blk * 64, q0, h, b);
          }
        }
        issued = w + 1;
      }
    }
  } else if (warp == 5) {
    // ---- score products of each half: S^T_h = K Q_h^T, dP^T_h = V dout_h^T --
    const uint32_t idesc_s = idesc_bf16_f32(128, 64, 0);
    bool ok = nw == 0 || __all_sync(0xffffffffu, mbar_wait(&bars->kv_full, 0, abort_flag));
    for (int w = 0; ok && w < nw; ++w) {
      const int s = w % C::kSlots, r = w / C::kSlots;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars->qd_full[s], r & 1, abort_flag)))) break;
      const uint32_t sq = smem_addr(qd_smem + 2 * s * Geo<D>::kTile);
      const uint32_t sdo = sq + Geo<D>::kTile;
      for (int h = 0; h < 2; ++h) {
        // half h's buffers: the gradient products of the previous tile's half h are done
        if (w >= 1 &&
            !(ok = __all_sync(0xffffffffu, mbar_wait(&bars->pd_free[h], (w - 1) & 1, abort_flag))))
          break;
        tc_fence_after();
        if (lane == 0) {
          // rows 64 h .. 64 h + 63 of each [128 x 64] block of Q and dout
          mma_scores<D>(tmem + C::kS + 64 * h, smem_addr(k_smem), sq + h * 64 * 128, idesc_s);
          tc_commit(&bars->s_full[h]);
          mma_scores<D>(tmem + C::kDp + 64 * h, smem_addr(v_smem), sdo + h * 64 * 128, idesc_s);
          tc_commit(&bars->dp_full[h]);
        }
        __syncwarp();
        last_commit = &bars->dp_full[h];
        last_parity = w & 1;
      }
    }
  } else if (warp == 6) {
    // ---- gradient products: dV += w^T_h dout_h, dK += dS^T_h Q_h ----------
    const uint32_t idesc_g = idesc_bf16_f32(128, D, 1);
    bool ok = true;
    for (int w = 0; ok && w < nw; ++w) {
      const int s = w % C::kSlots;
      const uint32_t sq = smem_addr(qd_smem + 2 * s * Geo<D>::kTile);
      const uint32_t sdo = sq + Geo<D>::kTile;
      for (int h = 0; h < 2; ++h) {
        // A: 16 queries = 8 packed columns; B: 16 query rows (MN-major).  dV
        // goes as soon as w^T_h is in TMEM, dK once dS^T_h is
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars->w_full[h], w & 1, abort_flag))))
          break;
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t rows = (h * 64 + kk * 16) * 128;
            const uint32_t acc = (w > 0 || h > 0 || kk > 0) ? 1u : 0u;
            tc_mma_ts(tmem + C::kDv, tmem + C::kS + 64 * h + kk * 8,
                      smem_desc_sw128(sdo + rows, Geo<D>::kBlk, 1024), idesc_g, acc);
          }
        }
        __syncwarp();
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bars->ds_full[h], w & 1, abort_flag))))
          break;
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t rows = (h * 64 + kk * 16) * 128;
            const uint32_t acc = (w > 0 || h > 0 || kk > 0) ? 1u : 0u;
            tc_mma_ts(tmem + C::kDk, tmem + C::kDp + 64 * h + kk * 8,
                      smem_desc_sw128(sq + rows, Geo<D>::kBlk, 1024), idesc_g, acc);
          }
          tc_commit(&bars->pd_free[h]);
          if (h == 1) tc_commit(&bars->qd_empty[s]);
        }
        __syncwarp();
        last_commit = &bars->pd_free[h];
        last_parity = w & 1;
      }
    }
    if (ok && nw > 0 && lane == 0) tc_commit(&bars->done);
    __syncwarp();
  } else {
    const int r = threadIdx.x;
    const int j = k0 + r;  // this thread's key
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    // queries [i_min, i_max) may read key j
    const bool key_ok = j < p.Lk && !((p.mask & kMaskKeyPadding) && j >= len);
    int i_min = 0, i_max = p.Lq;
    if (p.mask & kMaskCausal) i_min = j;
    if (p.mask & kMaskCausalTail) i_min = max(i_min, j - len + p.Lq);
    if (p.mask & kMaskQueryPadding) i_max = min(i_max, len);
    if (!key_ok) i_max = i_min;
    bool ok = true;
    for (int w = 0; ok && w < nw; ++w) {
      const int s = w % C::kSlots;
      const int q0 = (t_lo + w % per_head) * kT;
      const float *st = stat + s * (C::kStat / 4);
      for (int h = 0; h < 2; ++h) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[h], w & 1, abort_flag));
        // the lse and D the producer stored before arriving on qd_full
        if (ok && h == 0)
          ok = __all_sync(0xffffffffu,
                          mbar_wait(&bars->qd_full[s], (w / C::kSlots) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_t = tmem + lane_base + C::kS + 64 * h;
        const uint32_t dp_t = tmem + lane_base + C::kDp + 64 * h;
        const float *sth = st + h * 64;
        const int c0 = q0 + h * 64;  // first query of the half
        // w^T while dP^T_h is still being computed: both 32-column chunks
        // load from TMEM at once (one wait)
        float wv[2][32];
        {
          uint32_t sv[2][32];
          tmem_ld32(s_t, sv[0]);
          tmem_ld32(s_t + 32, sv[1]);
          tmem_wait_ld();
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            uint32_t pw[16];
            dkdv_w32(sv[ch], sth + ch * 32, i_min - (c0 + ch * 32), i_max - (c0 + ch * 32),
                     p.scale_log2, wv[ch], pw);
            tmem_st16(s_t + ch * 16, pw);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->w_full[h]);
        // dS^T = w^T (dP^T - D)
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->dp_full[h], w & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t pv[2][32];
          tmem_ld32(dp_t, pv[0]);
          tmem_ld32(dp_t + 32, pv[1]);
          tmem_wait_ld();
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            uint32_t pd[16];
            dkdv_ds32(wv[ch], pv[ch], sth + ch * 32, pd);
            tmem_st16(dp_t + ch * 16, pd);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->ds_full[h]);
      }
    }
    // warp-collective TMEM loads by every thread; keys inside the tensor stored
    const bool key = j < p.Lk;
    if (nw > 0 && ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->done, 0, abort_flag));
      tc_fence_after();
    }
    uint16_t *dkr = static_cast<uint16_t *>(a.dk) + (key ? row_at(p.layout, b, hk, j, p.Hkv, p.Lk, D) : 0);
    uint16_t *dvr = static_cast<uint16_t *>(a.dv) + (key ? row_at(p.layout, b, hk, j, p.Hkv, p.Lk, D) : 0);
#pragma unroll 1
    for (int ch = 0; ok && ch < D / 32; ++ch) {
      if (nw > 0) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + C::kDv + ch * 32, v);
        tmem_wait_ld();
        if (key) store_row32(dvr + ch * 32, v, 1.f);
        tmem_ld32(tmem + lane_base + C::kDk + ch * 32, v);
        tmem_wait_ld();
        if (key) store_row32(dkr + ch * 32, v, a.scale);
      } else if (key) {
        store_zero32(dvr + ch * 32);
        store_zero32(dkr + ch * 32);
      }
    }
  }

  if (*abort_flag && warp == 4 && lane == 0) {
    for (int idx = issued - C::kSlots; idx < issued; ++idx)
      if (idx >= 0) (void)wait_teardown(&bars->qd_full[idx % C::kSlots], (idx / C::kSlots) & 1);
    if (nw > 0) (void)wait_teardown(&bars->kv_full, 0);
  }
  if (*abort_flag && (warp == 5 || warp == 6) && lane == 0 && last_commit != nullptr)
    (void)wait_teardown(last_commit, last_parity);
  if (*abort_flag && threadIdx.x == 0) atomicExch(p.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, 512);
}

// ============================================================================
// short: query and key lengths of one tile (<= 128), d = 64 -- the whole
// backward of a unit of (batch, key/value head) pairs in one persistent CTA
// ============================================================================
// A unit holds a.pack pairs of one batch element (packed like the forward's
// short kernel: pair p in tile rows [p R, p R + R), R = 128 / pack; products
// between different pairs land in blocks that are masked to zero) or, with
// shared key/value heads, one pair and the query heads of its group.  Per
// query head (thread r of the softmax warpgroup owns tile row r):
//   S = Q K^T, dP = dout V^T          tcgen05.mma -> TMEM (rows on the lanes)
//   w = softmax(S) over the row's allowed keys (its one key tile gives the
//   exact statistics), dS = w (dP - D), D = dout . out
//   w, dS (bf16) -> shared memory, one [128 x 128] tile each in the 128-byte
//   swizzled layout (two 64-key slabs): read K-major it is the A operand
//   [queries x keys] of dQ = dS K, read MN-major the A operand [keys x
//   queries] of dV += w^T dout and dK += dS^T Q, so nothing is recomputed
//   with the keys on the lanes
// S and dP of head n + 1 go out as soon as the softmax has read those of head
// n, so the products of one head overlap the softmax of the next; the softmax
// stores dQ of head n (and dV, dK of a finished unit) after the exponentials
// of head n + 1, staged per warp so that each store instruction writes whole
// 64-byte row pieces.  D = dout . out comes from shared memory: dout from the
// head's TMA tile, out from rows each thread copies (cp.async) one head ahead
// -- a global load at the point of use stalled the softmax for microseconds.
// K and V of the next unit and Q and dout of the next head load while the
// current one computes.  TMEM: S | dP | dQ | dV | dK (448 columns).
// With the caller's row statistics (the forward's lse; kGiven, taken when the
// mask is not causal) the weights come straight from them, w = 2^(s scale
// log2(e) - lse), one 32-key chunk at a time, and a second warpgroup (warps
// 6-9) stores dQ, dV and dK, so the softmax warpgroup only forms w and dS.
// Otherwise the softmax warpgroup keeps its row of S in registers for the
// statistics and also stores.
struct ShortBwdBars {
  uint64_t kv_full[2], kv_empty[2];  // K, V of a unit (by unit parity)
  uint64_t qd_full[2], qd_empty[2];  // Q, dout of a head (by iteration parity)
  uint64_t sd_full;   // S, dP in TMEM
  uint64_t sd_free;   // S, dP read (softmax threads)
  uint64_t wd_full;   // w, dS in shared memory (softmax threads)
  uint64_t wd_free;   // the gradient products that read w, dS are done
  uint64_t dq_full;   // dQ in TMEM
  uint64_t dq_free;   // dQ read (softmax threads)
  uint64_t dkv_full;  // dV, dK of a unit complete
  uint64_t dkv_free;  // dV, dK read (softmax threads)
  uint64_t drain;     // teardown: the MMA thread's products have finished
  uint32_t tmem_base;
  int abort_flag;
};
constexpr int kSbTile = 128 * 128;  // one [128 x 64] bf16 tile
constexpr int kSbStage = 32 * 64;  // one softmax warp's 32 half-rows of output
// K, V (two units), Q, dout (two heads), w and dS (two 64-key slabs each),
// the rows of out, the softmax warps' output staging
constexpr size_t kSbSmem = 1024 + 13 * static_cast<size_t>(kSbTile) + 4 * kSbStage + 512;
constexpr uint32_t kSbS = 0, kSbDp = 128, kSbDq = 256, kSbDv = 320, kSbDk = 384;
// with the caller's statistics: softmax warpgroup (warps 0-3), producer (4),
// MMA issuer (5), stores (6-9)
constexpr int kSbThreadsGiven = 320;

// byte offset of 16-byte piece c (0..15: keys 8c .. 8c + 7) of row r in a
// [128 x 128] bf16 tile stored as two 128-byte-swizzled 64-key slabs
__device__ __forceinline__ uint32_t wd_offset(uint32_t r, uint32_t c) {
  return (c >> 3) * kSbTile + r * 128u + (((c & 7u) ^ (r & 7u)) << 4);
}
// byte offset of 16-byte piece c (0..3) of 64-byte half-row `row` (0..31) in
// a warp's staging buffer, swizzled so that the eight lanes of one shared
// memory wavefront never share a bank group, writing or reading
__device__ __forceinline__ uint32_t stage64(uint32_t row, uint32_t c) {
  return row * 64u + ((c ^ ((row >> 1) & 3u)) << 4);
}
// sum over 8 bf16 pairs of a[e] * b[e] (fp32)
__device__ __forceinline__ float dot_bf16x8(const uint4 &a, const uint4 &b) {
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
  float s = 0.f;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    s = fmaf(__uint_as_float(aw[t] << 16), __uint_as_float(bw[t] << 16), s);
    s = fmaf(__uint_as_float(aw[t] & 0xffff0000u), __uint_as_float(bw[t] & 0xffff0000u), s);
  }
  return s;
}

// w = 2^(s scale_log2 - lse) and dS = w (dP - D) over 32 key columns of the
// calling thread's row, packed to bf16 pairs: columns c in [lo, hi) are
// allowed, the others weigh 0.  A chunk the whole warp may read takes packed
// fp32 pairs, no mask.
__device__ __forceinline__ void short_chunk(const uint32_t (&sv)[32], const uint32_t (&pv)[32],
                                            int lo, int hi, float scale_log2, float lse, float dd,
                                            uint32_t (&pw)[16], uint32_t (&pd)[16]) {
  if (__all_sync(0xffffffffu, lo <= 0 && hi >= 32)) {
    const uint64_t sc = f2_pack(scale_log2, scale_log2), nl = f2_pack(-lse, -lse);
    const uint64_t d2 = f2_pack(dd, dd);
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      float x0, x1, g0, g1;
      f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), sc, nl),
                x0, x1);
      const float w0 = ex2_approx(x0), w1 = ex2_approx(x1);
      f2_unpack(f2_mul(f2_pack(w0, w1),
                       f2_sub(f2_pack(__uint_as_float(pv[e]), __uint_as_float(pv[e + 1])), d2)),
                g0, g1);
      pw[e >> 1] = pack_bf16x2(w0, w1);
      pd[e >> 1] = pack_bf16x2(g0, g1);
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    const float w0 =
        e >= lo && e < hi ? ex2_approx(__uint_as_float(sv[e]) * scale_log2 - lse) : 0.f;
    const float w1 =
        e + 1 >= lo && e + 1 < hi ? ex2_approx(__uint_as_float(sv[e + 1]) * scale_log2 - lse) : 0.f;
    pw[e >> 1] = pack_bf16x2(w0, w1);
    pd[e >> 1] = pack_bf16x2(w0 * (__uint_as_float(pv[e]) - dd),
                             w1 * (__uint_as_float(pv[e + 1]) - dd));
  }
}

template <bool kGiven>
__global__ void __launch_bounds__(kGiven ? kSbThreadsGiven : kThreads, 1)
    bwd_short_tc_kernel(const __grid_constant__ LongMaps maps, const Problem p, const BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *kv_smem = smem;                   // 2 x (K, V)
  uint8_t *qd_smem = kv_smem + 4 * kSbTile;  // 2 x (Q, dout)
  uint8_t *w_smem = qd_smem + 4 * kSbTile;   // w: two slabs
  uint8_t *ds_smem = w_smem + 2 * kSbTile;   // dS: two slabs
  uint8_t *out_smem = ds_smem + 2 * kSbTile;    // thread r: row r of out
  uint8_t *stage_smem = out_smem + kSbTile;     // 4 x 2 KiB output staging
  ShortBwdBars *bars = reinterpret_cast<ShortBwdBars *>(stage_smem + 4 * kSbStage);
  volatile int *abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int group = p.H / p.Hkv;
  const int P = a.pack, R = kT / a.pack;  // pairs per unit (1 when group > 1), rows per pair
  const int upb = (p.Hkv + P - 1) / P;    // units per batch element
  const int units = p.B * upb;
  const int G = static_cast<int>(gridDim.x);
  const int n_local = static_cast<int>(blockIdx.x) < units
                          ? (units - 1 - static_cast<int>(blockIdx.x)) / G + 1
                          : 0;
  const int n_it = n_local * group;  // (unit, query head) iterations of this CTA

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
      mbar_init(&bars->qd_full[i], 1);
      mbar_init(&bars->qd_empty[i], 1);
    }
    mbar_init(&bars->sd_full, 1);
    mbar_init(&bars->sd_free, kWg);
    mbar_init(&bars->wd_full, kWg);
    mbar_init(&bars->wd_free, 1);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, kWg);
    mbar_init(&bars->dkv_full, 1);
    mbar_init(&bars->dkv_free, kWg);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  int kv_issued = 0, qd_issued = 0;
  bool mma_issued = false;

  // ---- stores of dQ, dV, dK by a warp of the storing warpgroup: warp w
  // reads TMEM lanes [32 (w mod 4), + 32), i.e. those tile rows ------------
  const int quad = warp & 3;
  const uint32_t lane_q = static_cast<uint32_t>(quad * 32) << 16;
  const int rows_shift = __ffs(R) - 1;  // R is a power of two
  const uint32_t so = smem_addr(stage_smem + quad * kSbStage);
  // 32 TMEM columns of this thread's row (fp32) * f -> bf16 -> the warp's
  // staging; then the warp writes its 32 half-rows, eight 64-byte pieces per
  // store instruction.  dst(rr) is the global address of warp row rr's
  // half-row (nullptr: not stored).
  auto stage_store = [&](const uint32_t (&v)[32], float f, auto dst) {
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4)
      st_shared_v4(so + stage64(lane, c4),
                   pack_bf16x2(__uint_as_float(v[8 * c4 + 0]) * f, __uint_as_float(v[8 * c4 + 1]) * f),
                   pack_bf16x2(__uint_as_float(v[8 * c4 + 2]) * f, __uint_as_float(v[8 * c4 + 3]) * f),
                   pack_bf16x2(__uint_as_float(v[8 * c4 + 4]) * f, __uint_as_float(v[8 * c4 + 5]) * f),
                   pack_bf16x2(__uint_as_float(v[8 * c4 + 6]) * f, __uint_as_float(v[8 * c4 + 7]) * f));
    __syncwarp();
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int rr = 8 * t + (lane >> 2);
      const uint4 val = ld_shared_v4(so + stage64(rr, lane & 3));
      uint16_t *g = dst(rr);
      if (g != nullptr) st_global_v4(g + (lane & 3) * 8, val);
    }
    __syncwarp();
  };
  // dQ of iteration `it` (tile row: pair row >> rows_shift, query row & (R - 1))
  auto store_dq = [&](int it) -> bool {
    if (!__all_sync(0xffffffffu, mbar_wait(&bars->dq_full, it & 1, abort_flag))) return false;
    tc_fence_after();
    const int ul = it / group, hl = it - ul * group;
    const int u = static_cast<int>(blockIdx.x) + ul * G;
    const int b = u / upb, hk0 = (u - b * upb) * P;
    auto dst = [&](int ch) {
      return [&, ch](int rr) -> uint16_t * {
        const int row = quad * 32 + rr, pp = row >> rows_shift, i = row & (R - 1);
        return hk0 + pp < p.Hkv && i < p.Lq
                   ? static_cast<uint16_t *>(a.dq) +
                         row_at(p.layout, b, (hk0 + pp) * group + hl, i, p.H, p.Lq, 64) + ch * 32
                   : nullptr;
      };
    };
#pragma unroll 1
    for (int ch = 0; ch < 2; ++ch) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_q + kSbDq + ch * 32, v);
      tmem_wait_ld();
      stage_store(v, a.scale, dst(ch));
    }
    tc_fence_before();
    mbar_arrive(&bars->dq_free);
    return true;
  };
  // dV and dK of unit ul (tile row = key row: pair row >> rows_shift)
  auto store_dkv = [&](int ul) -> bool {
    const bool okd = __all_sync(0xffffffffu, mbar_wait(&bars->dkv_full, ul & 1, abort_flag));
    if (!named_barrier_and(1, kWg, okd)) return false;
    tc_fence_after();
    const int u = static_cast<int>(blockIdx.x) + ul * G;
    const int b = u / upb, hk0 = (u % upb) * P;
    // element offset of key row rr of this warp (or -1)
    auto key_at = [&](int rr) -> long long {
      const int row = quad * 32 + rr, pp = row >> rows_shift, j = row & (R - 1);
      return hk0 + pp < p.Hkv && j < p.Lk
                 ? static_cast<long long>(row_at(p.layout, b, hk0 + pp, j, p.Hkv, p.Lk, 64))
                 : -1LL;
    };
    auto dst = [&](void *base, int ch) {
      return [&, base, ch](int rr) -> uint16_t * {
        const long long o = key_at(rr);
        return o >= 0 ? static_cast<uint16_t *>(base) + o + ch * 32 : nullptr;
      };
    };
#pragma unroll 1
    for (int ch = 0; ch < 2; ++ch) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_q + kSbDv + ch * 32, v);
      tmem_wait_ld();
      stage_store(v, 1.f, dst(a.dv, ch));
      tmem_ld32(tmem + lane_q + kSbDk + ch * 32, v);
      tmem_wait_ld();
      stage_store(v, a.scale, dst(a.dk, ch));
    }
    tc_fence_before();
    mbar_arrive(&bars->dkv_free);
    return true;
  };

  if (warp == 4) {
    // ---- producer: per unit K and V, then Q and dout of each query head ----
    int it = 0;
    for (int ul = 0; ul < n_local; ++ul) {
      const int u = static_cast<int>(blockIdx.x) + ul * G;
      const int b = u / upb, hk0 = (u % upb) * P;
      const int kb = ul & 1;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&bars->kv_empty[kb], ((ul >> 1) & 1) ^ 1, abort_flag)))
        break;
      if (lane == 0) {
        uint8_t *dst = kv_smem + 2 * kb * kSbTile;
        mbar_arrive_expect_tx(&bars->kv_full[kb], 2 * kSbTile);
        tma_load_4d(dst, &maps.k, &bars->kv_full[kb], 0, 0, hk0, b);
        tma_load_4d(dst + kSbTile, &maps.v, &bars->kv_full[kb], 0, 0, hk0, b);
      }
      kv_issued = ul + 1;
      bool ok = true;
      for (int hl = 0; hl < group; ++hl, ++it) {
        const int st = it & 1;
        if (!(ok = __all_sync(0xffffffffu,
                              mbar_wait(&bars->qd_empty[st], ((it >> 1) & 1) ^ 1, abort_flag))))
          break;
        if (lane == 0) {
          uint8_t *dst = qd_smem + 2 * st * kSbTile;
          mbar_arrive_expect_tx(&bars->qd_full[st], 2 * kSbTile);
          tma_load_4d(dst, &maps.q, &bars->qd_full[st], 0, 0, hk0 * group + hl, b);
          tma_load_4d(dst + kSbTile, &maps.o, &bars->qd_full[st], 0, 0, hk0 * group + hl, b);
        }
        qd_issued = it + 1;
      }
      if (!ok) break;
    }
  } else if (warp == 5) {
    // ---- MMA issuer: S, dP of iteration n + 1 before the gradients of n ------
    const uint32_t idesc_s = idesc_bf16_f32(128, kT, 0);  // A, B K-major
    const uint32_t idesc_q = idesc_bf16_f32(128, 64, 1);  // A K-major, B MN-major
    const uint32_t idesc_kv = idesc_q | (1u << 15);       // A and B MN-major
    const uint32_t sw = smem_addr(w_smem), sds = smem_addr(ds_smem);
    auto wait = [&](uint64_t *bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
    };
    auto scores = [&](int it) -> bool {
      const int ul = it / group, hl = it - ul * group, kb = ul & 1, st = it & 1;
      if (hl == 0 && !wait(&bars->kv_full[kb], (ul >> 1) & 1)) return false;
      if (!wait(&bars->qd_full[st], (it >> 1) & 1)) return false;
      if (it >= 1 && !wait(&bars->sd_free, (it - 1) & 1)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t sk = smem_addr(kv_smem + 2 * kb * kSbTile), sv = sk + kSbTile;
        const uint32_t sq = smem_addr(qd_smem + 2 * st * kSbTile), sdo = sq + kSbTile;
        mma_scores<64>(tmem + kSbS, sq, sk, idesc_s);    // S = Q K^T
        mma_scores<64>(tmem + kSbDp, sdo, sv, idesc_s);  // dP = dout V^T
        tc_commit(&bars->sd_full);
      }
      __syncwarp();
      mma_issued = true;
      return true;
    };
    auto grads = [&](int it) -> bool {
      const int ul = it / group, hl = it - ul * group, kb = ul & 1, st = it & 1;
      if (!wait(&bars->wd_full, it & 1)) return false;
      if (it >= 1 && !wait(&bars->dq_free, (it - 1) & 1)) return false;
      // the unit's first head overwrites dV, dK: the previous unit's were read
      if (hl == 0 && ul >= 1 && !wait(&bars->dkv_free, (ul - 1) & 1)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t sk = smem_addr(kv_smem + 2 * kb * kSbTile);
        const uint32_t sq = smem_addr(qd_smem + 2 * st * kSbTile), sdo = sq + kSbTile;
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)
          // dQ = dS K: A = dS K-major (16 keys = 32 bytes of a slab row), B =
          // K MN-major (16 key rows = 2 KiB)
          tc_mma_ss(tmem + kSbDq,
                    smem_desc_sw128(sds + (kk >> 2) * kSbTile + (kk & 3) * 32, 16, 1024),
                    smem_desc_sw128(sk + kk * 2048, kSbTile, 1024), idesc_q, kk > 0);
        tc_commit(&bars->dq_full);
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk) {
          // dV += w^T dout, dK += dS^T Q: A MN-major (16 queries = 2 KiB; the
          // two 64-key slabs one tile apart), B MN-major
          const uint32_t acc = (hl > 0 || kk > 0) ? 1u : 0u;
          tc_mma_ss(tmem + kSbDv, smem_desc_sw128(sw + kk * 2048, kSbTile, 1024),
                    smem_desc_sw128(sdo + kk * 2048, kSbTile, 1024), idesc_kv, acc);
          tc_mma_ss(tmem + kSbDk, smem_desc_sw128(sds + kk * 2048, kSbTile, 1024),
                    smem_desc_sw128(sq + kk * 2048, kSbTile, 1024), idesc_kv, acc);
        }
        tc_commit(&bars->wd_free);
        tc_commit(&bars->qd_empty[st]);
        if (hl == group - 1) {
          tc_commit(&bars->kv_empty[kb]);
          tc_commit(&bars->dkv_full);
        }
      }
      __syncwarp();
      return true;
    };
    bool ok = n_it == 0 || scores(0);
    for (int it = 0; ok && it < n_it; ++it) {
      if (it + 1 < n_it && !(ok = scores(it + 1))) break;
      ok = grads(it);
    }
  } else if (kGiven && warp >= 6) {
    // ---- stores (with the caller's statistics): dQ of every head, then dV
    // and dK of a finished unit
    bool ok = true;
    for (int it = 0; ok && it < n_it; ++it) {
      ok = store_dq(it);
      if (ok && it % group == group - 1) ok = store_dkv(it / group);
    }
  } else {
    // ---- softmax: thread r = tile row r (pair r / R, query r % R); without
    // the caller's statistics also the stores, thread r = tile row r of the
    // queries (dQ) and of the keys (dV, dK) ----------------------------------
    const int r = threadIdx.x;
    const int pr = r / R, ri = r - pr * R;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t swr = smem_addr(w_smem), sdsr = smem_addr(ds_smem);
    // query row (b, head h, position i) of tile row `row` at iteration `it`;
    // `valid` says whether it exists
    struct RowAt {
      int b, h, i;
      bool valid;
    };
    // (batch, first key/value head, head within the group) of an iteration
    struct Iter {
      int b, hk0, hl;
    };
    auto iter_of = [&](int it) -> Iter {
      const int ul = it / group;
      const int u = static_cast<int>(blockIdx.x) + ul * G;
      Iter t;
      t.b = u / upb;
      t.hk0 = (u - t.b * upb) * P;
      t.hl = it - ul * group;
      return t;
    };
    const int r_shift = __ffs(R) - 1;  // R is a power of two
    auto row_of = [&](const Iter &t, int row) -> RowAt {
      const int pp = row >> r_shift;
      RowAt x;
      x.b = t.b;
      x.i = row & (R - 1);
      x.h = (t.hk0 + pp) * group + t.hl;  // pp == 0 when group > 1
      x.valid = t.hk0 + pp < p.Hkv && x.i < p.Lq;
      return x;
    };
    // this thread's row of out for iteration `it` -> its shared-memory row
    // (cp.async, in flight for a whole iteration: thread r alone touches
    // row r, so no other thread waits for it)
    const uint32_t orow = smem_addr(out_smem) + r * 128;
    auto fetch_out = [&](int it) {
      const RowAt x = row_of(iter_of(it), r);
      if (!x.valid) return;
      const uint16_t *src = static_cast<const uint16_t *>(a.out) +
                            row_at(p.layout, x.b, x.h, x.i, p.H, p.Lq, 64);
#pragma unroll
      for (int c = 0; c < 8; ++c) cp_async16(orow + ((c ^ (r & 7)) << 4), src + 8 * c);
      cp_async_commit();
    };
    // D = dout . out of this thread's row: out from its cp.async row, dout
    // from the TMA tile of the iteration's stage (same 128-byte swizzle)
    auto row_dsum = [&](int it, bool valid) -> float {
      cp_async_wait_all();
      if (!valid) return 0.f;
      const uint32_t drow = smem_addr(qd_smem + 2 * (it & 1) * kSbTile + kSbTile) + r * 128;
      float dd = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t off = (c ^ (r & 7)) << 4;
        dd += dot_bf16x8(ld_shared_v4(orow + off), ld_shared_v4(drow + off));
      }
      return dd;
    };

    if constexpr (kGiven) {
      // the caller's log2 softmax denominator of the row at iteration `it`
      // (loaded one iteration ahead)
      auto lse_of = [&](int it) -> float {
        const RowAt x = row_of(iter_of(it), r);
        return x.valid ? a.lse[(static_cast<size_t>(x.b) * p.H + x.h) * p.Lq + x.i] : INFINITY;
      };
      float lse_next = n_it > 0 ? lse_of(0) : INFINITY;
      bool ok = true;
      if (n_it > 0) fetch_out(0);
      for (int it = 0; ok && it < n_it; ++it) {
        const Iter itr = iter_of(it);
        const RowAt x = row_of(itr, r);
        const int len = clamp_len(p, x.b);
        // allowed tile columns [lo, hi): the row's own pair, keys j < jmax
        const int lo = pr * R;
        const int hi = lo + (x.valid ? row_limit(p, len, ri) : 0);
        const float lse = lse_next;
        if (it + 1 < n_it) lse_next = lse_of(it + 1);
        // D of the row: dout's tile has landed (its phase cannot move on
        // before this head's gradients are issued), out's row came by cp.async
        if (!(ok = __all_sync(0xffffffffu,
                              mbar_wait(&bars->qd_full[it & 1], (it >> 1) & 1, abort_flag))))
          break;
        const float dd = row_dsum(it, x.valid);
        if (it + 1 < n_it) fetch_out(it + 1);
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->sd_full, it & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_t = tmem + lane_base + kSbS, dp_t = tmem + lane_base + kSbDp;
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          uint32_t sv[2][32], pv[2][32], pw[2][16], pd[2][16];
          tmem_ld32(s_t + 64 * c2, sv[0]);
          tmem_ld32(s_t + 64 * c2 + 32, sv[1]);
          tmem_ld32(dp_t + 64 * c2, pv[0]);
          tmem_ld32(dp_t + 64 * c2 + 32, pv[1]);
          tmem_wait_ld();
          if (c2 == 1) {
            // every read of S and dP is done: the next head's may go out
            tc_fence_before();
            mbar_arrive(&bars->sd_free);
          }
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
            short_chunk(sv[cc], pv[cc], lo - 32 * (2 * c2 + cc), hi - 32 * (2 * c2 + cc),
                        p.scale_log2, lse, dd, pw[cc], pd[cc]);
          // the previous head's gradient products have read w and dS
          if (c2 == 0 && it >= 1 &&
              !(ok = __all_sync(0xffffffffu,
                                mbar_wait(&bars->wd_free, (it - 1) & 1, abort_flag))))
            break;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const uint32_t off = wd_offset(r, (2 * c2 + cc) * 4 + t);
              st_shared_v4(swr + off, pw[cc][4 * t], pw[cc][4 * t + 1], pw[cc][4 * t + 2],
                           pw[cc][4 * t + 3]);
              st_shared_v4(sdsr + off, pd[cc][4 * t], pd[cc][4 * t + 1], pd[cc][4 * t + 2],
                           pd[cc][4 * t + 3]);
            }
        }
        if (!ok) break;
        // generic-proxy stores, read by the tensor core (async proxy)
        fence_proxy_async_smem();
        mbar_arrive(&bars->wd_full);
      }
    } else {
      bool ok = true;
      if (n_it > 0) fetch_out(0);
      for (int it = 0; ok && it < n_it; ++it) {
        const int ul = it / group, hl = it - ul * group;
        const Iter itr = iter_of(it);
        const RowAt x = row_of(itr, r);
        const int len = clamp_len(p, x.b);
        // allowed tile columns [lo, hi): the row's own pair, keys j < jmax
        const int lo = pr * R;
        const int hi = lo + (x.valid ? row_limit(p, len, ri) : 0);
        // D of the row: dout's tile has landed (its phase cannot move on before
        // this head's gradients are issued), out's row came by cp.async
        if (!(ok = __all_sync(0xffffffffu,
                              mbar_wait(&bars->qd_full[it & 1], (it >> 1) & 1, abort_flag))))
          break;
        const float dd = row_dsum(it, x.valid);
        if (it + 1 < n_it) fetch_out(it + 1);
        // ---- the row's softmax over its allowed keys, dS over dP
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->sd_full, it & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) tmem_ld32(tmem + lane_base + kSbS + ch * 32, sr[ch]);
        tmem_wait_ld();
        const bool need_mask = __any_sync(0xffffffffu, lo > 0 || hi < kT);
        const bool pos = p.scale_log2 > 0.f;
        const float m = pos ? mask_max128(sr, need_mask, lo, hi) * p.scale_log2
                            : scale_mask_max128(sr, p.scale_log2, need_mask, lo, hi);
        const float l = pos ? exp2_fma_sum128(sr, p.scale_log2, m, m != -INFINITY)
                            : exp2_sum128(sr, m, m != -INFINITY);
        const float inv = l > 0.f ? 1.f / l : 0.f;
        // the previous head's dQ, and the previous unit's dV and dK
        if (it >= 1 && !(ok = store_dq(it - 1))) break;
        if (it >= 1 && hl == 0 && !(ok = store_dkv(ul - 1))) break;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t pv[32], pw[16], pd[16];
          tmem_ld32(tmem + lane_base + kSbDp + ch * 32, pv);
          tmem_wait_ld();
          if (ch == 3) {
            // every read of S and dP is done: the next head's may go out
            tc_fence_before();
            mbar_arrive(&bars->sd_free);
          }
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float w0 = __uint_as_float(sr[ch][e]) * inv;
            const float w1 = __uint_as_float(sr[ch][e + 1]) * inv;
            pw[e >> 1] = pack_bf16x2(w0, w1);
            pd[e >> 1] = pack_bf16x2(w0 * (__uint_as_float(pv[e]) - dd),
                                     w1 * (__uint_as_float(pv[e + 1]) - dd));
          }
          // the previous head's gradient products have read w and dS
          if (ch == 0 && it >= 1 &&
              !(ok = __all_sync(0xffffffffu, mbar_wait(&bars->wd_free, (it - 1) & 1, abort_flag))))
            break;
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const uint32_t off = wd_offset(r, ch * 4 + t);
            st_shared_v4(swr + off, pw[4 * t], pw[4 * t + 1], pw[4 * t + 2], pw[4 * t + 3]);
            st_shared_v4(sdsr + off, pd[4 * t], pd[4 * t + 1], pd[4 * t + 2], pd[4 * t + 3]);
          }
        }
        if (!ok) break;
        // generic-proxy stores, read by the tensor core (async proxy)
        fence_proxy_async_smem();
        mbar_arrive(&bars->wd_full);
      }
      if (ok && n_it > 0) ok = store_dq(n_it - 1) && store_dkv(n_local - 1);
    }
  }

  if (*abort_flag && warp == 4 && lane == 0) {
    for (int i = kv_issued - 2; i < kv_issued; ++i)
      if (i >= 0) (void)wait_teardown(&bars->kv_full[i & 1], (i >> 1) & 1);
    for (int i = qd_issued - 2; i < qd_issued; ++i)
      if (i >= 0) (void)wait_teardown(&bars->qd_full[i & 1], (i >> 1) & 1);
  }
  if (*abort_flag && warp == 5 && lane == 0 && mma_issued) {
    // tcgen05 ops of one thread complete in order: one more commit covers
    // every product issued before it
    tc_commit(&bars->drain);
    (void)wait_teardown(&bars->drain, 0);
  }
  if (*abort_flag && threadIdx.x == 0) atomicExch(p.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, 512);
}

template <typename K>
cudaError_t launch_one(K kernel, size_t smem, long long grid, const LongMaps &maps,
                       const Problem &p, const BwdArgs &a, cudaStream_t stream,
                       int threads = kThreads) {
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaError_t e =
      set_smem_once(reinterpret_cast<const void *>(kernel), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kernel<<<static_cast<unsigned>(grid), threads, smem, stream>>>(maps, p, a);
  return cudaGetLastError();
}

// D_i = dout_i . out_i per query row (bf16 tensors, fp32 sums): D / 8 lanes
// per row, 16 bytes of each tensor per lane and step, a shuffle tree per row
template <int D>
__global__ void __launch_bounds__(256) bwd_dsum_kernel(const Problem p, const BwdArgs a) {
  constexpr int kLanesPerRow = D / 8, kRowsPerWarp = 32 / kLanesPerRow;
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLanesPerRow, c = (lane % kLanesPerRow) * 8;
  const size_t rows = static_cast<size_t>(p.B) * p.H * p.Lq;
  const size_t warp0 = (blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x) >> 5;
  const size_t nwarps = (gridDim.x * static_cast<size_t>(blockDim.x)) >> 5;
  for (size_t r0 = warp0 * kRowsPerWarp; r0 < rows; r0 += nwarps * kRowsPerWarp) {
    const size_t row = r0 + sub;
    float s = 0.f;
    if (row < rows) {
      const int i = static_cast<int>(row % p.Lq);
      const size_t bh = row / p.Lq;
      const int b = static_cast<int>(bh / p.H), h = static_cast<int>(bh % p.H);
      const size_t at = row_at(p.layout, b, h, i, p.H, p.Lq, D) + c;
      const uint4 ov = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.out) + at);
      const uint4 gv = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.dout) + at);
      const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        s = fmaf(__uint_as_float(ow[t] << 16), __uint_as_float(gw[t] << 16), s);
        s = fmaf(__uint_as_float(ow[t] & 0xffff0000u), __uint_as_float(gw[t] & 0xffff0000u), s);
      }
    }
#pragma unroll
    for (int o = kLanesPerRow / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (row < rows && c == 0) a.dsum[row] = s;
  }
}

template <int D>
cudaError_t launch_bwd_tc_impl(const LongMaps &maps, const Problem &p, const BwdArgs &a,
                               cudaStream_t stream, bool have_lse) {
  static_assert(StatsCfg<D>::kSmem <= 232448 && DqCfg<D>::kSmem <= 232448 &&
                    DkdvCfg<D>::kSmem <= 232448,
                "shared memory budget");
  const long long nqb = (p.Lq + kT - 1) / kT, nkb = (p.Lk + kT - 1) / kT;
  const long long q_grid = nqb * p.B * p.H, k_grid = nkb * p.B * p.Hkv;
  cudaError_t e = cudaSuccess;
  if (have_lse) {
    // the row statistics came with the forward pass: only D is left to form
    const long long rows = static_cast<long long>(p.B) * p.H * p.Lq;
    const long long blocks = (rows + 63) / 64;  // grid-stride beyond 8192 blocks
    bwd_dsum_kernel<D><<<static_cast<unsigned>(blocks < 8192 ? blocks : 8192), 256, 0, stream>>>(p, a);
    e = cudaGetLastError();
  } else {
    e = launch_one(bwd_stats_tc_kernel<D>, StatsCfg<D>::kSmem, q_grid, maps, p, a, stream);
  }
  if (e != cudaSuccess) return e;
  e = launch_one(bwd_dq_tc_kernel<D>, DqCfg<D>::kSmem, q_grid, maps, p, a, stream);
  if (e != cudaSuccess) return e;
  return launch_one(bwd_dkdv_tc_kernel<D>, DkdvCfg<D>::kSmem, k_grid, maps, p, a, stream,
                    kDkdvThreads);
}

}  // namespace

cudaError_t launch_bwd_tc(const LongMaps &maps, const Problem &p, const BwdArgs &a, int num_sms,
                          cudaStream_t stream, bool have_lse) {
  if (p.dk == 128) return launch_bwd_tc_impl<128>(maps, p, a, stream, have_lse);
  if (p.Lq <= kT && p.Lk <= kT) {
    // one tile each way: the fused persistent kernel (no statistics pass)
    const long long units = static_cast<long long>(p.B) * ((p.Hkv + a.pack - 1) / a.pack);
    const long long grid = units < num_sms ? units : num_sms;
    // the storing warpgroup pays where a row's softmax is heavy; under a
    // causal mask half of the keys are masked and the softmax warpgroup is
    // quicker doing its own stores (about 10% faster and 2% slower
    // respectively, measured on GB300)
    if (have_lse && !(p.mask & kMaskCausal))
      return launch_one(bwd_short_tc_kernel<true>, kSbSmem, grid, maps, p, a, stream,
                        kSbThreadsGiven);
    return launch_one(bwd_short_tc_kernel<false>, kSbSmem, grid, maps, p, a, stream);
  }
  return launch_bwd_tc_impl<64>(maps, p, a, stream, have_lse);
}

}  // namespace mha
