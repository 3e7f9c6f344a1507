// Packed short-sequence attention on the tcgen05 tensor cores (bf16, d = 64).
//
// Sentence-length attention (Lq, Lk <= 128) is bound by HBM traffic, not by
// arithmetic: each (batch, head) pair is one small Q K^T and one small P V.
// This kernel packs P = 128 / max(Rq, Rk) pairs into one 128-row tile (Rq,
// Rk: Lq, Lk rounded up to powers of two) so one tcgen05.mma covers all of
// them; products between different pairs land in off-diagonal blocks that the
// mask discards.  Each CTA is persistent (one per SM) and walks the units
// u = blockIdx.x, + gridDim.x, ...
//
// Warp roles (192 threads):
//   warps 0-3  softmax + epilogue, thread t owns tile row t
//   warp  4    TMA producer: Q, K, V of a unit into a 3-stage ring
//   warp  5    TMEM owner and MMA issuer
// Per unit (the four steps of scaled dot-product attention):
//   S = Q K^T              tcgen05.mma -> TMEM (fp32), double-buffered
//   mask, scale, softmax   tcgen05.ld -> registers; exp2 against the row max
//   P (bf16) -> smem       128-byte swizzled K-major operand
//   O = P V                tcgen05.mma -> TMEM (fp32), double-buffered
//   O / rowsum -> bf16     tcgen05.ld, swizzled smem tile, TMA store
// Padded sequences load only their first ceil(len/8)*8 rows (8-row TMA boxes),
// so padding costs no HBM reads; masked keys get exactly zero weight; padded
// query rows and rows without any allowed key are stored as +0.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kD = 64;
constexpr int kStages = 3;
constexpr int kTileRows = 128;
constexpr int kTileBytes = kTileRows * kD * 2;  // 16 KiB per operand tile
constexpr int kStageBytes = 3 * kTileBytes;     // Q | K | V
constexpr int kPBytes = kTileRows * 128 * 2;     // P tile: 128 x 128 bf16 (2 swizzle blocks)
constexpr int kThreads = 192;
constexpr int kSoftmaxThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol0 = 0;    // S buffers: cols [0,128), [128,256)
constexpr uint32_t kOCol0 = 256;  // O buffers: cols [256,320), [320,384)

struct __align__(8) Barriers {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t o_free[2];
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t kSmemBytes = 1024 /* alignment slack */ + kStages * kStageBytes + 2 * kPBytes +
                              sizeof(Barriers);

__device__ __forceinline__ int clamp_len(const Problem &p, int b) {
  if (!(p.mask & (kMaskKeyPadding | kMaskQueryPadding))) return p.Lk;
  const int l = p.key_lengths[b];
  return l < 0 ? 0 : (l > p.Lk ? p.Lk : l);
}

__device__ __forceinline__ bool wait_teardown(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity))
    if (global_timer_ns() - t0 > 100000000ull) return false;
  return true;
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_short_tc_kernel(const __grid_constant__ ShortMaps maps, const ShortGeom g,
                         const Problem p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *stage_base = smem;
  uint8_t *pbuf_base = smem + kStages * kStageBytes;
  Barriers *bars = reinterpret_cast<Barriers *>(pbuf_base + 2 * kPBytes);
  volatile int *abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BH = p.B * p.H;
  const int n_local = (static_cast<int>(blockIdx.x) < g.units)
                          ? (g.units - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1
                          : 0;

  // ---- setup -------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->p_full[b], kSoftmaxThreads);
      mbar_init(&bars->pv_done[b], 1);
      mbar_init(&bars->o_free[b], kSoftmaxThreads);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&maps.q_full);
    tma_prefetch_desc(&maps.k_full);
    tma_prefetch_desc(&maps.v_full);
    tma_prefetch_desc(&maps.o_store);
  }
  if (warp == 5) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // Rows that a padded unit does not load keep earlier contents; start from
  // zeros so they are always finite (their weights are exactly zero).
  for (int i = threadIdx.x; i < kStages * kStageBytes / 16; i += kThreads)
    reinterpret_cast<uint4 *>(stage_base)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  int issued = 0;                        // producer: units whose loads were issued
  uint64_t *last_commit = nullptr;       // MMA issuer: barrier of the last commit
  uint32_t last_commit_parity = 0;
  if (warp == 4) {
    // ---- TMA producer ----------------------------------------------------
    // lengths of the pairs of unit n, loaded one unit ahead of their use
    auto load_lens = [&](int n, int (&lens)[16]) {
      const int bh0 = (blockIdx.x + n * gridDim.x) * g.P;
#pragma unroll
      for (int pp = 0; pp < 16; ++pp)
        lens[pp] = (n < n_local && pp < g.P && bh0 + pp < BH) ? clamp_len(p, (bh0 + pp) / p.H) : 0;
    };
    int lens[16], lens_next[16];
    load_lens(0, lens);
    for (int n = 0; n < n_local; ++n) {
      const int s = n % kStages;
      const int u = blockIdx.x + n * gridDim.x;
      const int bh0 = u * g.P;
      load_lens(n + 1, lens_next);
      if (!mbar_wait(&bars->empty[s], ((n / kStages) & 1) ^ 1, abort_flag)) break;
      uint8_t *sq = stage_base + s * kStageBytes;
      uint8_t *sk = sq + kTileBytes;
      uint8_t *sv = sk + kTileBytes;
      // byte count of everything this unit loads
      uint32_t bytes = 0;
      if (!g.rows_q) bytes += g.P * g.Rq * 128;
      if (!g.rows_k) bytes += 2 * g.P * g.Rk * 128;
#pragma unroll
      for (int pp = 0; pp < 16; ++pp) {
        if (g.rows_q) bytes += ((min(lens[pp], p.Lq) + 7) / 8) * 1024;
        if (g.rows_k) bytes += 2 * ((lens[pp] + 7) / 8) * 1024;
      }
      if (lane == 0) mbar_arrive_expect_tx(&bars->full[s], bytes);
      __syncwarp();
      if (lane == 0) {
        if (!g.rows_q) tma_load_3d(sq, &maps.q_full, &bars->full[s], 0, 0, bh0);
        if (!g.rows_k) {
          tma_load_3d(sk, &maps.k_full, &bars->full[s], 0, 0, bh0);
          tma_load_3d(sv, &maps.v_full, &bars->full[s], 0, 0, bh0);
        }
      }
      if (g.rows_q || g.rows_k) {
        // 8-row boxes, spread over the lanes: item = (pair, box)
        const int boxes_per_pair = (g.Rq > g.Rk ? g.Rq : g.Rk) / 8;
        for (int it = lane; it < g.P * boxes_per_pair; it += 32) {
          const int pp = it / boxes_per_pair, bx = it % boxes_per_pair;
          int len_pp = 0;
#pragma unroll
          for (int t = 0; t < 16; ++t)
            if (t == pp) len_pp = lens[t];
          if (bh0 + pp >= BH) continue;
          const int r0 = bx * 8;
          if (g.rows_q && r0 < min(len_pp, p.Lq))
            tma_load_3d(sq + (pp * g.Rq + r0) * 128, &maps.q_rows, &bars->full[s], 0, r0,
                        bh0 + pp);
          if (g.rows_k && r0 < len_pp) {
            tma_load_3d(sk + (pp * g.Rk + r0) * 128, &maps.k_rows, &bars->full[s], 0, r0,
                        bh0 + pp);
            tma_load_3d(sv + (pp * g.Rk + r0) * 128, &maps.v_rows, &bars->full[s], 0, r0,
                        bh0 + pp);
          }
        }
      }
      __syncwarp();
      issued = n + 1;
#pragma unroll
      for (int pp = 0; pp < 16; ++pp) lens[pp] = lens_next[pp];
    }
  } else if (warp == 5) {
    // ---- MMA issuer (lane 0) ----------------------------------------------
    const uint32_t n_keys = static_cast<uint32_t>(g.P * g.Rk);  // multiple of 16, <= 128
    const uint32_t idesc_s = idesc_bf16_f32(128, n_keys, 0);
    const uint32_t idesc_o = idesc_bf16_f32(128, kD, 1);
    auto issue_s = [&](int n) -> bool {
      const int s = n % kStages, b = n & 1;
      if (!mbar_wait(&bars->full[s], (n / kStages) & 1, abort_flag)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t sq = smem_addr(stage_base + s * kStageBytes);
        const uint32_t sk = sq + kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint64_t da = smem_desc_sw128(sq + kk * 32, 16, 1024);
          const uint64_t db = smem_desc_sw128(sk + kk * 32, 16, 1024);
          tc_mma_ss(tmem + kSCol0 + b * 128, da, db, idesc_s, kk > 0);
        }
        tc_commit(&bars->s_full[b]);
      }
      __syncwarp();
      last_commit = &bars->s_full[b];
      last_commit_parity = (n >> 1) & 1;
      return true;
    };
    // Issue whichever product is ready first: S for the next unit (its data
    // landed, its S buffer is free) or P V for the oldest unit whose P is
    // written.  Neither waits behind the other.
    int ns = 0, npv = 0;
    uint64_t t_idle = 0;
    while (npv < n_local) {
      bool progressed = false;
      bool ready_s = false;
      if (ns < n_local && ns <= npv + 1 && lane == 0)
        ready_s = mbar_probe(&bars->full[ns % kStages], (ns / kStages) & 1);
      if (__shfl_sync(0xffffffffu, ready_s, 0)) {
        if (!issue_s(ns)) break;
        ++ns;
        progressed = true;
      }
      bool ready_pv = false;
      if (npv < ns && lane == 0)
        ready_pv = mbar_probe(&bars->p_full[npv & 1], (npv >> 1) & 1) &&
                   mbar_probe(&bars->o_free[npv & 1], ((npv >> 1) & 1) ^ 1);
      if (__shfl_sync(0xffffffffu, ready_pv, 0)) {
        const int s = npv % kStages, b = npv & 1;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sv = smem_addr(stage_base + s * kStageBytes + 2 * kTileBytes);
          const uint32_t sp = smem_addr(pbuf_base + b * kPBytes);
          for (uint32_t kk = 0; kk < n_keys / 16; ++kk) {
            // A = P (K-major, key block kk/4 of 64 keys, 32-byte step inside it)
            const uint64_t da = smem_desc_sw128(
                sp + (kk >> 2) * (kTileRows * 128) + (kk & 3) * 32, 16, 1024);
            // B = V (MN-major: 16 key rows per step, 64 value columns)
            const uint64_t db = smem_desc_sw128(sv + kk * 16 * 128, 1024, 1024);
            tc_mma_ss(tmem + kOCol0 + b * kD, da, db, idesc_o, kk > 0);
          }
          tc_commit(&bars->pv_done[b]);
          tc_commit(&bars->empty[s]);
        }
        __syncwarp();
        last_commit = &bars->empty[s];
        last_commit_parity = (npv / kStages) & 1;
        ++npv;
        progressed = true;
      }
      if (progressed) {
        t_idle = 0;
      } else {
        const uint64_t now = global_timer_ns();
        if (t_idle == 0) t_idle = now;
        if (*abort_flag) break;
        if (now - t_idle > kWaitLimitNs) {
          *abort_flag = 1;
          break;
        }
      }
    }
  } else {
    // ---- softmax + epilogue (warps 0-3; thread = tile row) -----------------
    const int r = threadIdx.x;
    const int pr = r / g.Rq, i = r % g.Rq;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;


    auto len_of = [&](int n) -> int {
      const int bh = (blockIdx.x + n * gridDim.x) * g.P + pr;
      const bool valid = pr < g.P && bh < BH && i < p.Lq;
      return valid ? clamp_len(p, bh / p.H) : 0;
    };
    int len_cur = n_local > 0 ? len_of(0) : 0;
    float rowsum_prev = 0.f;  // row sum of the unit whose epilogue is pending
    bool pending_zero = true;
    for (int n = 0; n <= n_local; ++n) {
      float rowsum = 0.f;
      bool zero_row = true;
      const int len_next = n + 1 < n_local ? len_of(n + 1) : 0;  // load ahead of its use
      if (n < n_local) {
        const int b = n & 1;
        const int u = blockIdx.x + n * gridDim.x;
        const int bh = u * g.P + pr;
        const bool valid = pr < g.P && bh < BH && i < p.Lq;
        const int len = len_cur;
        int jmax = p.Lk;
        if (p.mask & kMaskKeyPadding) jmax = min(jmax, len);
        if (p.mask & kMaskCausal) jmax = min(jmax, i + 1);
        const bool qpad = (p.mask & kMaskQueryPadding) && i >= len;
        if (!valid || qpad) jmax = 0;
        const int col_lo = pr * g.Rk;

        if (!mbar_wait(&bars->s_full[b], (n >> 1) & 1, abort_flag)) break;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
          tmem_ld32(tmem + lane_base + kSCol0 + b * 128 + ch * 32, sr[ch]);
        tmem_wait_ld();
        tc_fence_before();
        // scale (log2 units), keep only this row's keys [col_lo, col_lo + jmax)
        const float m = scale_mask_max128(sr, p.scale_log2, true, col_lo, col_lo + jmax);
        const bool any = m != -INFINITY;
        rowsum = exp2_sum128(sr, m, any);
        zero_row = !any;

        // the P buffer b was last the staging tile of unit n-2's output store
        if (threadIdx.x == 0) tma_store_wait_read0();
        named_barrier_sync(1, kSoftmaxThreads);
        const uint32_t sp = smem_addr(pbuf_base + b * kPBytes);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {  // 16-byte pieces of 8 columns
            uint32_t w[4];
#pragma unroll
            for (int t = 0; t < 4; ++t)
              w[t] = pack_bf16x2(__uint_as_float(sr[ch][q4 * 8 + 2 * t]),
                                 __uint_as_float(sr[ch][q4 * 8 + 2 * t + 1]));
            const int c16 = ch * 4 + q4;  // 0..15
            const uint32_t addr =
                sp + (c16 >> 3) * (kTileRows * 128) + sw128_offset(r, c16 & 7);
            st_shared_v4(addr, w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars->p_full[b]);
      }
      // epilogue of unit n-1 (its P V product ran while we did unit n)
      if (n >= 1) {
        const int pn = n - 1, b = pn & 1;
        const int u = blockIdx.x + pn * gridDim.x;
        if (!mbar_wait(&bars->pv_done[b], (pn >> 1) & 1, abort_flag)) break;
        tc_fence_after();
        uint32_t o[2][32];
        tmem_ld32(tmem + lane_base + kOCol0 + b * kD, o[0]);
        tmem_ld32(tmem + lane_base + kOCol0 + b * kD + 32, o[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars->o_free[b]);
        const float inv = pending_zero ? 0.f : 1.f / rowsum_prev;
        // stage the bf16 row in the (now free) P buffer b, 128-byte swizzled
        const uint32_t so = smem_addr(pbuf_base + b * kPBytes);
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          uint32_t w[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int c = c8 * 8 + 2 * t;
            const float a0 = pending_zero ? 0.f : __uint_as_float(o[c >> 5][c & 31]) * inv;
            const float a1 =
                pending_zero ? 0.f : __uint_as_float(o[(c + 1) >> 5][(c + 1) & 31]) * inv;
            w[t] = pack_bf16x2(a0, a1);
          }
          st_shared_v4(so + sw128_offset(r, c8), w[0], w[1], w[2], w[3]);
        }
        fence_proxy_async_smem();
        named_barrier_sync(1, kSoftmaxThreads);
        if (threadIdx.x == 0) {
          tma_store_3d(&maps.o_store, pbuf_base + b * kPBytes, 0, 0, u * g.P);
          tma_store_commit();
        }
      }
      rowsum_prev = rowsum;
      pending_zero = zero_row;
      len_cur = len_next;
    }
    if (threadIdx.x == 0) tma_store_wait0();
  }

  // ---- teardown ------------------------------------------------------------
  if (*abort_flag && warp == 4 && lane == 0) {
    // let copies already in flight land before the CTA's shared memory goes away
    for (int n = issued - kStages; n < issued; ++n)
      if (n >= 0) (void)wait_teardown(&bars->full[n % kStages], (n / kStages) & 1);
  }
  if (*abort_flag && warp == 5 && lane == 0 && last_commit != nullptr) {
    // tcgen05 ops complete in order: the last commit covers all of them
    (void)wait_teardown(last_commit, last_commit_parity);
  }
  if (*abort_flag && threadIdx.x == 0) atomicExch(p.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_short_tc(const ShortMaps &maps, const ShortGeom &g, const Problem &p,
                            int num_sms, cudaStream_t stream) {
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(attn_short_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const int grid = g.units < num_sms ? g.units : num_sms;
  if (grid <= 0) return cudaSuccess;
  attn_short_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(maps, g, p);
  return cudaGetLastError();
}

}  // namespace mha
