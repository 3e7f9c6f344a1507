// y = x W + b on the tcgen05 tensor cores (bf16 in, fp32 accumulate, bf16 out).
//
// The learned projections of the multi-head sublayer: x [M, K] row-major
// (token vectors), W [K, N] row-major (input-major, as in Q · W^Q with W^Q of
// shape d_model x d_k), b [N], y [M, N] row-major.
//
// Persistent: one CTA per SM walks 128 x 128 output tiles (all N tiles of an
// M block before the next M block, so the x block is reused from L2).
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

template <bool kSlabs>
__global__ void __launch_bounds__(kThreads, 1)
    linear_tc_kernel(const __grid_constant__ LinearMaps maps, const uint16_t *__restrict__ bias,
                     uint16_t *__restrict__ y, int M, int N, int K, int *status) {
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
  const int n_tiles_n = (N + kBN - 1) / kBN;
  const int n_tiles = ((M + kBM - 1) / kBM) * n_tiles_n;
  const int n_kb = (K + kBK - 1) / kBK;

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
    tma_prefetch_desc(&maps.x);
    tma_prefetch_desc(&maps.w);
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
        const int m0 = (t / n_tiles_n) * kBM, n0 = (t % n_tiles_n) * kBN;
        const bool second = n0 + 64 < N;  // the tile's second 64-column block exists
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int s = it % kStages;
          if (!(ok = mbar_wait(&bars->empty[s], ((it / kStages) & 1) ^ 1, abort_flag))) break;
          uint8_t *sa = smem + s * kStageBytes;
          uint8_t *sb = sa + kATile;
          if (kSlabs) {
            // boxes past the matrix edges fill with zeros and still count
            mbar_arrive_expect_tx(&bars->full[s], kStageBytes);
            tma_load_3d(sa, &maps.x, &bars->full[s], 0, m0, kb * 2);
            tma_load_3d(sb, &maps.w, &bars->full[s], 0, kb * kBK, n0 / 64);
          } else {
            mbar_arrive_expect_tx(&bars->full[s], kATile + (second ? kBTile : kBBlock));
            tma_load_2d(sa, &maps.x, &bars->full[s], kb * kBK, m0);
            tma_load_2d(sb, &maps.w, &bars->full[s], n0, kb * kBK);
            if (second) tma_load_2d(sb + kBBlock, &maps.w, &bars->full[s], n0 + 64, kb * kBK);
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
      if (!(ok = mbar_wait(&bars->acc_empty[a], ((tl >> 1) & 1) ^ 1, abort_flag))) break;
      tc_fence_after();
      for (int kb = 0; kb < n_kb; ++kb, ++it) {
        const int s = it % kStages;
        if (!(ok = mbar_wait(&bars->full[s], (it / kStages) & 1, abort_flag))) break;
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
    const int q = warp & 3;  // TMEM lane quadrant of this warp
    const int e = warp - 2;  // epilogue warp index: staging and bias slots
    const uint32_t so = smem_addr(staging + e * kStagingBytes);
    float *bs = bias_s + e * kBN;
    int tl = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++tl) {
      const int a = tl & 1;
      const int m0 = (t / n_tiles_n) * kBM, n0 = (t % n_tiles_n) * kBN;
      // the tile's bias, as fp32, in this warp's slot (zeros past N or
      // without a bias)
#pragma unroll
      for (int c = lane; c < kBN; c += 32)
        bs[c] = (bias != nullptr && n0 + c < N)
                    ? __uint_as_float(static_cast<uint32_t>(bias[n0 + c]) << 16)
                    : 0.f;
      __syncwarp();
      if (!mbar_wait(&bars->acc_full[a], (tl >> 1) & 1, abort_flag)) break;
      tc_fence_after();
      const uint32_t tacc = tmem + (static_cast<uint32_t>(q * 32) << 16) + a * kBN;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t v[2][32];
        tmem_ld32(tacc + 64 * h, v[0]);
        tmem_ld32(tacc + 64 * h + 32, v[1]);
        tmem_wait_ld();
        if (h == 1) {
          tc_fence_before();
          mbar_arrive(&bars->acc_empty[a]);
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
          if (row < M && col < N)
            st_global_v4(y + static_cast<long long>(row) * N + col, val);
        }
        __syncwarp();
      }
    }
  }

  // ---- teardown ------------------------------------------------------------
  if (*abort_flag && warp == 0 && lane == 0) {
    for (int i = issued - kStages; i < issued; ++i)
      if (i >= 0) (void)wait_teardown(&bars->full[i % kStages], (i / kStages) & 1);
  }
  if (*abort_flag && warp == 1 && lane == 0 && last_commit != nullptr)
    (void)wait_teardown(last_commit, last_parity);
  if (*abort_flag && threadIdx.x == 0) atomicExch(status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_linear_tc(const LinearMaps &maps, const void *bias, void *y, int M, int N,
                             int K, bool slabs, int *status, int num_sms, cudaStream_t stream) {
  static_assert(Tiling<true>::kSmem <= 232448 && Tiling<false>::kSmem <= 232448,
                "shared memory budget");
  static_assert(Tiling<true>::kStages <= kMaxStages && Tiling<false>::kStages <= kMaxStages,
                "barrier slots");
  auto kernel = slabs ? linear_tc_kernel<true> : linear_tc_kernel<false>;
  const size_t smem = slabs ? Tiling<true>::kSmem : Tiling<false>::kSmem;
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(kernel), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long tiles =
      static_cast<long long>((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
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
  return cudaLaunchKernelEx(&cfg, kernel, maps,
                            static_cast<const uint16_t *>(bias), static_cast<uint16_t *>(y), M,
                            N, K, status);
}

}  // namespace mha
