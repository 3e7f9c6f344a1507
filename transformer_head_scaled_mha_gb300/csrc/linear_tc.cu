// y = x W + b on the tcgen05 tensor cores (bf16 in, fp32 accumulate, bf16 out).
//
// The learned projections of the multi-head sublayer: x [M, K] row-major
// (token vectors), W [K, N] row-major (input-major, as in Q · W^Q with W^Q of
// shape d_model x d_k), b [N], y [M, N] row-major.  One launch computes up to
// three such products with the same K (the query, key and value projections
// of a sublayer), each with its own x, W, b, y, M and N.
//
// Persistent: one CTA per SM walks the 128 x 128 output tiles of the products
// one after the other (all N tiles of an M block before the next M block, so
// the x block is reused from L2).
// Warp roles (192 threads):
//   warp 0      TMA producer: per K block an x tile [128 rows x K block]
//               (K-major, 128-byte swizzle) and a W tile [K block x 128
//               columns] as two 64-column blocks (MN-major), into a ring
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma (M128 N128 K16) per
//               16 of K into one of two TMEM accumulators (128 columns each),
//               so a tile's epilogue overlaps the next tile's products
//   warps 2-5   epilogue: thread = tile row; fp32 accumulator + bias -> bf16,
//               staged per warp (32 rows x 64 columns, swizzled) and written
//               with stores that each cover four whole 128-byte row pieces
// Rows, columns and K beyond the matrix edges read as zeros (TMA fill) and
// are never stored.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kBM = 128, kBN = 128;
constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kStagingBytes = 32 * 128;        // one warp's 32 rows x 64 columns
constexpr uint32_t kTmemCols = 256;            // two 128-column accumulators

constexpr int kMaxStages = 6;
struct __align__(8) Barriers {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint32_t tmem_base;
  int abort_flag;
};

// Two tilings of the K loop.  Slabs (K and N multiples of 64): a stage is a
// 128-wide K block, loaded as two 64-wide swizzle slabs per operand with one
// 3-D TMA box each (x viewed as (64, M, K/64), W as (64, K, N/64)); the copy
// engine spends a fixed cost per box, so fewer, larger boxes feed the tensor
// pipe faster (measured 15-21% over the 2-D tiling).  Otherwise a stage is a
// 64-wide K block with 2-D boxes, which handles any K, N multiple of 8.
template <bool kSlabs>
struct Tiling {
  static constexpr int kBK = kSlabs ? 128 : 64;
  static constexpr int kStages = kSlabs ? 3 : 6;
  static constexpr int kATile = kBM * kBK * 2;        // x: [128 rows x kBK]
  static constexpr int kBBlock = kBK * 64 * 2;        // W: kBK rows x 64 columns
  static constexpr int kBTile = 2 * kBBlock;
  static constexpr int kStageBytes = kATile + kBTile;  // 64 or 32 KiB
  static constexpr size_t kSmem = 1024 /* alignment slack */ + kStages * kStageBytes +
                                  kEpiWarps * kStagingBytes + kEpiWarps * kBN * 4 +
                                  sizeof(Barriers);
};

// The products of one launch: tiles [tiles_end[g - 1], tiles_end[g]) are
// product g's, n-tile-major within an M block.
struct LinearArgs {
  const uint16_t *bias[kMaxLinear];  // or nullptr
  uint16_t *y[kMaxLinear];
  int M[kMaxLinear], N[kMaxLinear];
  int tiles_n[kMaxLinear];    // N tiles of product g
  int tiles_end[kMaxLinear];  // one past product g's last tile
  int count, K;
  int *status;
};

// product, M offset and N offset of tile t (tiles bn columns wide)
struct TileAt {
  int g, m0, n0;
};
template <int bn = kBN>
__device__ __forceinline__ TileAt tile_at(const LinearArgs &a, int t) {
  TileAt x;
  x.g = t < a.tiles_end[0] ? 0 : (t < a.tiles_end[1] ? 1 : 2);
  const int lt = t - (x.g > 0 ? a.tiles_end[x.g - 1] : 0);
  const int tn = a.tiles_n[x.g];
  x.m0 = (lt / tn) * kBM;
  x.n0 = (lt - (lt / tn) * tn) * bn;
  return x;
}

// Epilogue of one 128 x 128 tile by warps 2-5 (thread = tile row): waits for
// its accumulator (phase `tl` / 2 of `full`), adds the bias, rounds to bf16,
// stages each warp's 32 rows x 64 columns (swizzled) and writes them with
// stores that each cover four whole 128-byte row pieces; frees the
// accumulator (`empty`) once it is read.  False when the wait gave up.
__device__ __forceinline__ bool epilogue_tile(const LinearArgs &args, const TileAt &at,
                                              uint64_t *full, int tl, uint32_t tacc_col,
                                              uint64_t *empty, uint32_t so, float *bs,
                                              volatile int *abort_flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;  // TMEM lane quadrant of this warp
  const int m0 = at.m0, n0 = at.n0, M = args.M[at.g], N = args.N[at.g];
  const uint16_t *bias = args.bias[at.g];
  uint16_t *y = args.y[at.g];
  // the tile's bias, as fp32, in this warp's slot (zeros past N or without a
  // bias)
#pragma unroll
  for (int c = lane; c < kBN; c += 32)
    bs[c] = (bias != nullptr && n0 + c < N)
                ? __uint_as_float(static_cast<uint32_t>(bias[n0 + c]) << 16)
                : 0.f;
  __syncwarp();
  if (!mbar_wait(full, (tl >> 1) & 1, abort_flag)) return false;
  tc_fence_after();
  const uint32_t tacc = tacc_col + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    uint32_t v[2][32];
    tmem_ld32(tacc + 64 * h, v[0]);
    tmem_ld32(tacc + 64 * h + 32, v[1]);
    tmem_wait_ld();
    if (h == 1 && empty != nullptr) {
      tc_fence_before();
      mbar_arrive(empty);
    }
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      uint32_t wv[4];
#pragma unroll
      for (int t2 = 0; t2 < 4; ++t2) {
        const int c = c8 * 8 + 2 * t2;
        wv[t2] = pack_bf16x2(__uint_as_float(v[c >> 5][c & 31]) + bs[64 * h + c],
                             __uint_as_float(v[c >> 5][(c + 1) & 31]) + bs[64 * h + c + 1]);
      }
      st_shared_v4(so + sw128_offset(lane, c8), wv[0], wv[1], wv[2], wv[3]);
    }
    __syncwarp();
    // four rows x 128 bytes per store instruction
#pragma unroll
    for (int t2 = 0; t2 < 8; ++t2) {
      const int rr = 4 * t2 + (lane >> 3);
      const int row = m0 + q * 32 + rr;
      const int col = n0 + 64 * h + (lane & 7) * 8;
      const uint4 val = ld_shared_v4(so + sw128_offset(rr, lane & 7));
      if (row < M && col < N) st_global_v4(y + static_cast<long long>(row) * N + col, val);
    }
    __syncwarp();
  }
  return true;
}

template <bool kSlabs>
__global__ void __launch_bounds__(kThreads, 1)
    linear_tc_kernel(const __grid_constant__ LinearMaps maps, const __grid_constant__ LinearArgs args) {
  using C = Tiling<kSlabs>;
  constexpr int kBK = C::kBK, kStages = C::kStages, kATile = C::kATile,
                kBBlock = C::kBBlock, kBTile = C::kBTile, kStageBytes = C::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *staging = smem + kStages * kStageBytes;
  float *bias_s = reinterpret_cast<float *>(staging + kEpiWarps * kStagingBytes);
  Barriers *bars = reinterpret_cast<Barriers *>(bias_s + kEpiWarps * kBN);
  volatile int *abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = args.tiles_end[args.count - 1];
  const int n_kb = (args.K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars->acc_full[a], 1);
      mbar_init(&bars->acc_empty[a], kEpiWarps * 32);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int g = 0; g < args.count; ++g) {
      tma_prefetch_desc(&maps.x[g]);
      tma_prefetch_desc(&maps.w[g]);
    }
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  griddep_wait();
  griddep_launch_dependents();

  int issued = 0;  // producer: K blocks whose loads were issued
  uint64_t *last_commit = nullptr;
  uint32_t last_parity = 0;
  if (warp == 0) {
    // ---- TMA producer -------------------------------------------------------
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        const TileAt tl = tile_at(args, t);
        const int m0 = tl.m0, n0 = tl.n0;
        const CUtensorMap *mx = &maps.x[tl.g], *mw = &maps.w[tl.g];
        // the tile's second 64-column block exists
        const bool second = n0 + 64 < args.N[tl.g];
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int s = it % kStages;
          if (!(ok = mbar_wait_spin(&bars->empty[s], ((it / kStages) & 1) ^ 1, abort_flag, kWaitLimitNs))) break;
          uint8_t *sa = smem + s * kStageBytes;
          uint8_t *sb = sa + kATile;
          if (kSlabs) {
            // boxes past the matrix edges fill with zeros and still count
            mbar_arrive_expect_tx(&bars->full[s], kStageBytes);
            tma_load_3d(sa, mx, &bars->full[s], 0, m0, kb * 2);
            tma_load_3d(sb, mw, &bars->full[s], 0, kb * kBK, n0 / 64);
          } else {
            mbar_arrive_expect_tx(&bars->full[s], kATile + (second ? kBTile : kBBlock));
            tma_load_2d(sa, mx, &bars->full[s], kb * kBK, m0);
            tma_load_2d(sb, mw, &bars->full[s], n0, kb * kBK);
            if (second) tma_load_2d(sb + kBBlock, mw, &bars->full[s], n0 + 64, kb * kBK);
          }
          issued = it + 1;
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer ---------------------------------------------------------
    const uint32_t idesc = idesc_bf16_f32(kBM, kBN, 1);  // B (W) is MN-major
    int it = 0, tl = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++tl) {
      const int a = tl & 1;
      if (!(ok = mbar_wait_spin(&bars->acc_empty[a], ((tl >> 1) & 1) ^ 1, abort_flag, kWaitLimitNs))) break;
      tc_fence_after();
      for (int kb = 0; kb < n_kb; ++kb, ++it) {
        const int s = it % kStages;
        if (!(ok = mbar_wait_spin(&bars->full[s], (it / kStages) & 1, abort_flag, kWaitLimitNs))) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sa = smem_addr(smem + s * kStageBytes);
          const uint32_t sb = sa + kATile;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            // A: 16 K columns = 32 bytes along a swizzled row (64 per slab, the
            // slabs kATile / 2 apart); B: 16 K rows = 2 KiB, its two 64-column
            // blocks kBBlock apart
            tc_mma_ss(tmem + a * kBN,
                      smem_desc_sw128(sa + (kk >> 2) * (kATile / 2) + (kk & 3) * 32, 16, 1024),
                      smem_desc_sw128(sb + kk * 16 * 128, kBBlock, 1024), idesc, kb > 0 || kk > 0);
          tc_commit(&bars->empty[s]);
          if (kb == n_kb - 1) tc_commit(&bars->acc_full[a]);
        }
        __syncwarp();
        last_commit = kb == n_kb - 1 ? &bars->acc_full[a] : &bars->empty[s];
        last_parity = kb == n_kb - 1 ? (tl >> 1) & 1 : (it / kStages) & 1;
      }
    }
  } else {
    // ---- epilogue -----------------------------------------------------------
    const int e = warp - 2;  // epilogue warp index: staging and bias slots
    const uint32_t so = smem_addr(staging + e * kStagingBytes);
    float *bs = bias_s + e * kBN;
    int tl = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++tl) {
      const int a = tl & 1;
      const TileAt at = tile_at(args, t);
      if (!epilogue_tile(args, at, &bars->acc_full[a], tl, tmem + a * kBN, &bars->acc_empty[a],
                         so, bs, abort_flag))
        break;
    }
  }

  // ---- teardown ------------------------------------------------------------
  if (*abort_flag && warp == 0 && lane == 0) {
    for (int i = issued - kStages; i < issued; ++i)
      if (i >= 0) (void)wait_teardown(&bars->full[i % kStages], (i / kStages) & 1);
  }
  if (*abort_flag && warp == 1 && lane == 0 && last_commit != nullptr)
    (void)wait_teardown(last_commit, last_parity);
  if (*abort_flag && threadIdx.x == 0) atomicExch(args.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ============================================================================
// Wide tiles (K and every N multiples of 64, N >= 256): 128 x 256 output
// tiles, one M128 N256 product per 16 of K.  A stage is 64 of K: x [128 x 64]
// (16 KiB) and W [64 x 256] as four 64-column slabs (32 KiB), so per output
// element the SM takes in 3/4 of the operand bytes of the 128 x 128 tiling --
// with K = 512 that tiling is bound by how fast operands reach the SM, not by
// the tensor core.  TMEM: two 256-column accumulators.
// ============================================================================
constexpr int kWN = 256;
constexpr int kWA = kBM * 64 * 2;        // 16 KiB
constexpr int kWB = 64 * kWN * 2;        // 32 KiB: 4 slabs of [64 rows x 64 columns]
constexpr int kWSlab = 64 * 128;         // one slab, 8 KiB
constexpr int kWStages = 4;
struct __align__(8) WideBarriers {
  uint64_t full[kWStages], empty[kWStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;  // teardown: every product of the CTA has finished
  uint32_t tmem_base;
  int abort_flag;
};
constexpr size_t kWSmem = 1024 + kWStages * (kWA + kWB) + kEpiWarps * kStagingBytes +
                          kEpiWarps * kWN * 4 + sizeof(WideBarriers);


__global__ void __launch_bounds__(kThreads, 1)
    linear_wide_kernel(const __grid_constant__ LinearMaps maps,
                       const __grid_constant__ LinearArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *staging = smem + kWStages * (kWA + kWB);
  float *bias_s = reinterpret_cast<float *>(staging + kEpiWarps * kStagingBytes);
  WideBarriers *bars = reinterpret_cast<WideBarriers *>(bias_s + kEpiWarps * kWN);
  volatile int *abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = args.tiles_end[args.count - 1];
  const int n_kb = args.K / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars->acc_full[a], 1);
      mbar_init(&bars->acc_empty[a], kEpiWarps * 32);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int g = 0; g < args.count; ++g) {
      tma_prefetch_desc(&maps.x[g]);
      tma_prefetch_desc(&maps.w[g]);
    }
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 2 * kWN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  griddep_wait();
  griddep_launch_dependents();

  int issued = 0;  // producer: stages whose loads were issued
  bool mma_issued = false;
  if (warp == 0) {
    // ---- TMA producer -------------------------------------------------------
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        const TileAt at = tile_at<kWN>(args, t);
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int s = it % kWStages;
          if (!(ok = mbar_wait_spin(&bars->empty[s], ((it / kWStages) & 1) ^ 1, abort_flag, kWaitLimitNs))) break;
          uint8_t *sa = smem + s * (kWA + kWB);
          // boxes past the matrix edges fill with zeros and still count
          mbar_arrive_expect_tx(&bars->full[s], kWA + kWB);
          tma_load_3d(sa, &maps.x[at.g], &bars->full[s], 0, at.m0, kb);
          tma_load_3d(sa + kWA, &maps.w[at.g], &bars->full[s], 0, kb * 64, at.n0 / 64);
          issued = it + 1;
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer ---------------------------------------------------------
    const uint32_t idesc = idesc_bf16_f32(kBM, kWN, 1);  // B (W) is MN-major
    int it = 0, tl = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++tl) {
      const int a = tl & 1;
      if (!(ok = mbar_wait_spin(&bars->acc_empty[a], ((tl >> 1) & 1) ^ 1, abort_flag, kWaitLimitNs))) break;
      tc_fence_after();
      for (int kb = 0; kb < n_kb; ++kb, ++it) {
        const int s = it % kWStages;
        if (!(ok = mbar_wait_spin(&bars->full[s], (it / kWStages) & 1, abort_flag, kWaitLimitNs))) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sa = smem_addr(smem + s * (kWA + kWB)), sb = sa + kWA;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            // A: 16 K columns = 32 bytes of a swizzled row; B: 16 K rows =
            // 2 KiB of each slab, the four 64-column slabs kWSlab apart
            tc_mma_ss(tmem + a * kWN, smem_desc_sw128(sa + kk * 32, 16, 1024),
                      smem_desc_sw128(sb + kk * 2048, kWSlab, 1024), idesc, kb > 0 || kk > 0);
          tc_commit(&bars->empty[s]);
          if (kb == n_kb - 1) tc_commit(&bars->acc_full[a]);
        }
        __syncwarp();
        mma_issued = true;
      }
    }
  } else {
    // ---- epilogue: the two 128-column halves of a tile as two 128 x 128 ----
    const int e = warp - 2;
    const uint32_t so = smem_addr(staging + e * kStagingBytes);
    float *bs = bias_s + e * kWN;
    int tl = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++tl) {
      const int a = tl & 1;
      const TileAt at = tile_at<kWN>(args, t);
      bool ok = true;
      for (int hh = 0; ok && hh < 2; ++hh) {
        TileAt half = at;
        half.n0 = at.n0 + hh * kBN;
        // the accumulator is free after the second half's reads; the first
        // half arrives on a barrier nobody waits for (the drain barrier's
        // phase never completes during the run)
        ok = epilogue_tile(args, half, &bars->acc_full[a], tl, tmem + a * kWN + hh * kBN,
                           hh == 1 ? &bars->acc_empty[a] : nullptr, so, bs + hh * kBN,
                           abort_flag);
      }
      if (!ok) break;
    }
  }

  // ---- teardown ------------------------------------------------------------
  if (*abort_flag && warp == 0 && lane == 0) {
    for (int i = issued - kWStages; i < issued; ++i)
      if (i >= 0) (void)wait_teardown(&bars->full[i % kWStages], (i / kWStages) & 1);
  }
  if (*abort_flag && warp == 1 && lane == 0 && mma_issued) {
    tc_commit(&bars->drain);
    (void)wait_teardown(&bars->drain, 0);
  }
  if (*abort_flag && threadIdx.x == 0) atomicExch(args.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 2 * kWN);
}

}  // namespace

bool linear_wide(int K, bool slabs, int min_n) { return slabs && K % 64 == 0 && min_n >= kWN; }

cudaError_t launch_linear_tc(const LinearMaps &maps, const LinearProblem *probs, int count,
                             int K, bool slabs, int *status, int num_sms, cudaStream_t stream) {
  static_assert(Tiling<true>::kSmem <= 232448 && Tiling<false>::kSmem <= 232448,
                "shared memory budget");
  static_assert(Tiling<true>::kStages <= kMaxStages && Tiling<false>::kStages <= kMaxStages,
                "barrier slots");
  if (count < 1 || count > kMaxLinear) return cudaErrorInvalidValue;
  int min_n = probs[0].N;
  for (int g = 1; g < count; ++g) min_n = probs[g].N < min_n ? probs[g].N : min_n;
  const bool wide = linear_wide(K, slabs, min_n);
  LinearArgs a;
  std::memset(&a, 0, sizeof a);
  long long tiles = 0;
  for (int g = 0; g < count; ++g) {
    a.bias[g] = static_cast<const uint16_t *>(probs[g].bias);
    a.y[g] = static_cast<uint16_t *>(probs[g].y);
    a.M[g] = probs[g].M;
    a.N[g] = probs[g].N;
    a.tiles_n[g] = (probs[g].N + (wide ? kWN : kBN) - 1) / (wide ? kWN : kBN);
    tiles += static_cast<long long>((probs[g].M + kBM - 1) / kBM) * a.tiles_n[g];
    if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
    a.tiles_end[g] = static_cast<int>(tiles);
  }
  for (int g = count; g < kMaxLinear; ++g) a.tiles_end[g] = static_cast<int>(tiles);
  a.count = count;
  a.K = K;
  a.status = status;
  static_assert(kWSmem <= 232448, "shared memory budget");
  auto kernel = wide ? linear_wide_kernel
                     : (slabs ? linear_tc_kernel<true> : linear_tc_kernel<false>);
  const size_t smem = wide ? kWSmem : (slabs ? Tiling<true>::kSmem : Tiling<false>::kSmem);
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kernel), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (tiles <= 0) return cudaSuccess;
  const int grid = tiles < num_sms ? static_cast<int>(tiles) : num_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, maps, a);
}

}  // namespace mha
