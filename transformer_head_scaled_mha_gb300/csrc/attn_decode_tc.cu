// Attention of a few query rows against a long key/value cache on the
// tcgen05 tensor cores (bf16, d in {64, 128}): the decoding step of
// generation, where each new token attends to every cached key of its
// sequence (trishampatil.com, "Scaled Dot-Product Attention: Step by Step",
// with the decoder's causal masking of alexdo.xyz, "Decoder block", applied to
// the last Lq positions as in "How predictions are generated").
//
// Work unit: one (batch element b, key/value head g) pair and its
// R = group x Lq query rows -- the `group` query heads that share key/value
// head g, Lq positions each, row r = (head within the group) * Lq + position;
// R <= 16.  Persistent CTAs, one per SM, each take a contiguous range of
// pairs holding an equal share of the work (key tiles plus a fixed cost per
// pair; lengths read on the device);
// the K/V stream runs ahead across pair boundaries.
//
// With so few query rows, the usual orientation (query rows on the 128 TMEM
// lanes, one thread per row) would leave most threads idle and put all 128
// exponentials of a tile row on one thread.  The scores are computed
// transposed instead, keys on the lanes:
//
//   S^T = K_j Q^T        tcgen05.mma M=128 keys, N=16 query rows, K=d; A = the
//                        K tile, B = Q, both K-major in 128B-swizzled smem;
//                        fp32 accumulator in TMEM
//   softmax              thread k holds key k's scores for every query row;
//                        a row's tile maximum is a warp shuffle reduction plus
//                        a 4-warp exchange in smem; the running maximum moves
//                        only when it grows by more than 2^8 (numerator and
//                        denominator share the stale maximum, so the quotient
//                        is unchanged), and O is rescaled in TMEM when it does;
//                        each thread keeps partial row sums for its key slot
//   P -> smem (bf16)     P over the tile's 128 keys, 16 rows per 64-key half
//                        (K-major, 128B swizzle)
//   O^T += V_j^T P^T     tcgen05.mma, A = the V tile read MN-major, B = P.
//                        d = 128: M = 128 value dims, N = 16, 8 key steps.
//                        d = 64: both 64-key halves of the tile in one product
//                        -- M rows 0..63 take the first half's values, 64..127
//                        the second half's (A's second M block lies 64 key
//                        rows further), N = 32 takes the first half's P rows
//                        then the second's; the two diagonal blocks of D are
//                        partial outputs over the two halves, summed at the
//                        end: 4 key steps per tile instead of 8
//   epilogue             row sums reduced over the 128 threads, O^T read from
//                        TMEM (thread = value dim), O / l -> bf16 -> global
//
// Pipelining: S is double-buffered in TMEM (S_{t+1} is computed while the
// softmax works on S_t), P in smem, and O and Q per pair (a pair's epilogue
// overlaps the next pair).  With products this small the issuing thread, not
// the tensor core, sets the pace, so two warps issue: one the score products
// S_t (once the softmax has read S_{t-2}), the other the PV products (as soon
// as P_t is written).  The softmax overwrites P buffer t % 2 only after PV_{t-2}
// has completed; every wait on a per-parity PV barrier is then at most one
// phase behind.  The softmax loops are compiled for RP = R rounded up to a
// power of two (rows R..RP-1 masked), so a one-row step does one row's work.
//
// Warp roles (224 threads): warps 0-3 softmax and epilogue, warp 4 TMA
// producer, warp 5 TMEM owner and score-product issuer, warp 6 PV issuer.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kThreads = 224;
constexpr int kSoftmaxThreads = 128;
constexpr int kBN = 128;            // keys per tile
constexpr int kN = 16;              // query rows per score product (R <= kN)
constexpr uint32_t kTmemCols = 128;  // S0 S1 (kN each), O0 O1 (kOCols each)
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kMaxSlots = 6;
constexpr uint32_t kBarSoftmax = 1;  // named barrier of the softmax warps

template <int D>
struct Cfg {
  static constexpr int kBlkBytes = 128 * 128;              // [128 rows x 64] swizzle block
  static constexpr int kTileBytes = (D / 64) * kBlkBytes;  // a K or V tile
  static constexpr int kSlotBytes = 2 * kTileBytes;        // ring slot: K tile, V tile
  static constexpr int kSlots = D == 128 ? 3 : 6;
  static constexpr int kQBlk = kN * 128;                   // [16 rows x 64] of Q or P
  static constexpr int kQBytes = (D / 64) * kQBlk;         // Q buffer
  static constexpr int kPBytes = 2 * kQBlk;                // P buffer: 16 rows x 128 keys
  static constexpr int kPvN = D == 64 ? 32 : 16;           // N of the PV product
  static constexpr int kPvSteps = D == 64 ? 4 : 8;         // its key steps
  // A's second M block: d = 64, the tile's keys 64..127 (64 rows down);
  // d = 128, value dims 64..127 (the next swizzle block)
  static constexpr uint32_t kVLbo = D == 64 ? 64 * 128 : kBlkBytes;
  static constexpr int kOCols = kPvN;
};

struct __align__(16) Shared {
  float red[2][4][kN];  // per-warp tile maxima, double-buffered by tile
  float lsum[4][kN];    // per-warp row sums
  float xo[kN][64];     // d = 64: the second key half's partial output
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[kMaxSlots], kv_empty[kMaxSlots];
  uint64_t s_full[2];   // S_t in TMEM
  uint64_t p_full[2];   // P_t in smem, S_t read (softmax threads)
  uint64_t pv_done[2];  // PV_t done, by tile parity
  uint64_t o_free[2];   // the epilogue has read O of a pair
  uint32_t tmem_base;
  int abort_flag;
};

template <int D>
constexpr size_t smem_bytes() {
  using C = Cfg<D>;
  return 1024 + static_cast<size_t>(C::kSlots) * C::kSlotBytes + 2 * C::kQBytes +
         2 * C::kPBytes + sizeof(Shared);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// key length of batch element b, clamped to [0, Lk]
__device__ __forceinline__ int key_len(const Problem &p, int b) {
  if (!(p.mask & kMaskKeyPadding)) return p.Lk;
  const int l = p.key_lengths[b];
  return l < 0 ? 0 : (l > p.Lk ? p.Lk : l);
}

// Cost of a pair in half-tile units: its key tiles plus a fixed 1.5 tiles
// for the pair's own work (Q load, row sums, output), which costs about that
// much when pairs are short.
__device__ __forceinline__ int pair_cost(int tiles) { return 2 * tiles + 3; }

// This CTA's pairs [lo, hi).  Pair (b, g) = b * Hkv + g starts at
// s = Hkv * (cost of the batch elements' pairs before b) + g * cost(b) in the
// concatenation of all pairs' costs, T in all; CTA c takes the pairs whose
// start lies in [ceil(c T / G), ceil((c + 1) T / G)) -- contiguous ranges whose
// costs differ by at most one pair's.  The whole warp calls it and gets the
// same answer in every lane.
__device__ void pair_range(const Problem &p, int lane, int &lo, int &hi) {
  const long long G = gridDim.x, c = blockIdx.x;
  const int npairs = p.B * p.Hkv;
  if (!(p.mask & kMaskKeyPadding)) {  // equal pairs
    lo = static_cast<int>((c * npairs + G - 1) / G);
    hi = static_cast<int>(((c + 1) * npairs + G - 1) / G);
    return;
  }
  long long total = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    const int t = b < p.B ? pair_cost((key_len(p, b) + kBN - 1) / kBN) : 0;
    total += __reduce_add_sync(0xffffffffu, static_cast<unsigned>(t));
  }
  total *= p.Hkv;
  const long long x_lo = (c * total + G - 1) / G, x_hi = ((c + 1) * total + G - 1) / G;
  lo = npairs;
  hi = npairs;
  bool found_lo = false, found_hi = c == G - 1;
  long long carry = 0;  // s of the first pair of this chunk of batch elements
  for (int b0 = 0; b0 < p.B && !(found_lo && found_hi); b0 += 32) {
    const int b = b0 + lane;
    const int t = b < p.B ? pair_cost((key_len(p, b) + kBN - 1) / kBN) : 0;
    int inc = t;  // inclusive scan of the pair costs over the chunk
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    const long long s0 = carry + static_cast<long long>(p.Hkv) * (inc - t);  // s(b, 0)
    // first head g of b whose pair starts at or after x (Hkv: none)
    auto first_g = [&](long long x) -> int {
      if (b >= p.B) return p.Hkv;
      if (s0 >= x) return 0;
      const long long g = (x - s0 + t - 1) / t;
      return g < p.Hkv ? static_cast<int>(g) : p.Hkv;
    };
    const int g_lo = first_g(x_lo), g_hi = first_g(x_hi);
    const unsigned m_lo = __ballot_sync(0xffffffffu, g_lo < p.Hkv);
    const unsigned m_hi = __ballot_sync(0xffffffffu, g_hi < p.Hkv);
    if (!found_lo && m_lo != 0) {
      const int f = __ffs(m_lo) - 1;
      lo = (b0 + f) * p.Hkv + __shfl_sync(0xffffffffu, g_lo, f);
      found_lo = true;
    }
    if (!found_hi && m_hi != 0) {
      const int f = __ffs(m_hi) - 1;
      hi = (b0 + f) * p.Hkv + __shfl_sync(0xffffffffu, g_hi, f);
      found_hi = true;
    }
    carry += static_cast<long long>(p.Hkv) * __shfl_sync(0xffffffffu, inc, 31);
  }
}

// Lane l: the key length of pair n0 + l (0 past hi).
__device__ __forceinline__ int pair_lens(const Problem &p, int n0, int hi, int lane) {
  const int pair = n0 + lane;
  return pair < hi ? key_len(p, pair / p.Hkv) : 0;
}

template <int D, int RP>
__global__ void __launch_bounds__(kThreads, 1)
    attn_decode_tc_kernel(const __grid_constant__ DecodeMaps maps, const Problem p,
                          uint16_t *__restrict__ out) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *ring = smem;                              // kSlots (K tile, V tile)
  uint8_t *qbuf = ring + C::kSlots * C::kSlotBytes;  // 2 Q buffers
  uint8_t *pbuf = qbuf + 2 * C::kQBytes;             // 2 P buffers
  Shared *sh = reinterpret_cast<Shared *>(pbuf + 2 * C::kPBytes);
  volatile int *abort_flag = &sh->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int group = p.H / p.Hkv;
  const int R = group * p.Lq;
  const bool tail = (p.mask & kMaskCausalTail) != 0;

  // ---- setup -------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh->q_full[i], 1);
      mbar_init(&sh->q_empty[i], 1);
      mbar_init(&sh->s_full[i], 1);
      mbar_init(&sh->p_full[i], kSoftmaxThreads);
      mbar_init(&sh->pv_done[i], 1);
      mbar_init(&sh->o_free[i], kSoftmaxThreads);
    }
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(&sh->kv_full[s], 1);
      mbar_init(&sh->kv_empty[s], 1);
    }
    sh->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(&sh->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  griddep_launch_dependents();

  int issued = 0, q_issued = 0;  // producer: K/V and Q loads issued
  uint64_t *last_commit = nullptr;
  uint32_t last_parity = 0;

  if (warp == 4) {
    // ---- TMA producer: per pair Q, then (K_j, V_j) through the ring --------
    if (lane == 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
    }
    griddep_wait();
    int lo, hi;
    pair_range(p, lane, lo, hi);
    bool ok = true;
    int lens = 0;
    for (int pair = lo; pair < hi && ok; ++pair) {
      const int n = pair - lo;
      if ((n & 31) == 0) lens = pair_lens(p, pair, hi, lane);
      const int len = __shfl_sync(0xffffffffu, lens, n & 31);
      const int nt = (len + kBN - 1) / kBN;
      if (nt == 0) continue;
      const int b = pair / p.Hkv, g = pair - b * p.Hkv;
      const int qb = q_issued & 1;
      ok = __all_sync(0xffffffffu,
                      mbar_wait(&sh->q_empty[qb], ((q_issued >> 1) & 1) ^ 1, abort_flag));
      if (!ok) break;
      if (lane == 0) {
        // the group's query heads, all Lq positions: R rows of 128 bytes
        mbar_arrive_expect_tx(&sh->q_full[qb], static_cast<uint32_t>((D / 64) * R * 128));
        for (int blk = 0; blk < D / 64; ++blk)
          tma_load_4d(qbuf + qb * C::kQBytes + blk * C::kQBlk, &maps.q, &sh->q_full[qb],
                      blk * 64, 0, g * group, b);
      }
      ++q_issued;
      for (int j = 0; j < nt; ++j) {
        const int slot = issued % C::kSlots, round = issued / C::kSlots;
        ok = __all_sync(0xffffffffu, mbar_wait(&sh->kv_empty[slot], (round & 1) ^ 1, abort_flag));
        if (!ok) break;
        if (lane == 0) {
          uint8_t *dst = ring + slot * C::kSlotBytes;
          mbar_arrive_expect_tx(&sh->kv_full[slot], C::kSlotBytes);
          for (int blk = 0; blk < D / 64; ++blk)
            tma_load_4d(dst + blk * C::kBlkBytes, &maps.k, &sh->kv_full[slot], blk * 64, j * kBN,
                        g, b);
          for (int blk = 0; blk < D / 64; ++blk)
            tma_load_4d(dst + C::kTileBytes + blk * C::kBlkBytes, &maps.v, &sh->kv_full[slot],
                        blk * 64, j * kBN, g, b);
        }
        ++issued;
      }
    }
  } else if (warp == 5) {
    // ---- score products S_t = K_t Q^T (lane 0 issues; the warp waits) -----
    const uint32_t idesc_s = idesc_bf16_f32(128, kN, 0);
    griddep_wait();
    int lo, hi;
    pair_range(p, lane, lo, hi);
    bool ok = true;
    int t = 0, qi = 0, slot = 0, round = 0;
    int lens = 0;
    for (int pair = lo; pair < hi && ok; ++pair) {
      const int n = pair - lo;
      if ((n & 31) == 0) lens = pair_lens(p, pair, hi, lane);
      const int len = __shfl_sync(0xffffffffu, lens, n & 31);
      const int nt = (len + kBN - 1) / kBN;
      if (nt == 0) continue;
      const int qb = qi & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&sh->q_full[qb], (qi >> 1) & 1, abort_flag));
      for (int j = 0; j < nt && ok; ++j) {
        ok = __all_sync(0xffffffffu, mbar_wait(&sh->kv_full[slot], round & 1, abort_flag));
        // S buffer t % 2 held S_{t-2}: the softmax has read it once P_{t-2} is out
        if (ok && t >= 2)
          ok = __all_sync(0xffffffffu,
                          mbar_wait(&sh->p_full[t & 1], ((t - 2) >> 1) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint64_t da0 = smem_desc_sw128(smem_addr(ring + slot * C::kSlotBytes), 16, 1024);
          const uint64_t db0 = smem_desc_sw128(smem_addr(qbuf + qb * C::kQBytes), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = (kk >> 2) * C::kBlkBytes + (kk & 3) * 32;
            const uint32_t kb = (kk >> 2) * C::kQBlk + (kk & 3) * 32;
            tc_mma_ss(tmem + (t & 1) * kN, da0 + (ka >> 4), db0 + (kb >> 4), idesc_s,
                      kk > 0 ? 1u : 0u);
          }
          tc_commit(&sh->s_full[t & 1]);
          if (j == nt - 1) tc_commit(&sh->q_empty[qb]);
        }
        __syncwarp();
        last_commit = &sh->s_full[t & 1];
        last_parity = (t >> 1) & 1;
        ++t;
        if (++slot == C::kSlots) {
          slot = 0;
          ++round;
        }
      }
      ++qi;
    }
  } else if (warp == 6) {
    // ---- PV products O (+)= P_t V_t (lane 0 issues; the warp waits) --------
    const uint32_t idesc_o = idesc_bf16_f32_amn(128, C::kPvN, 0);
    griddep_wait();
    int lo, hi;
    pair_range(p, lane, lo, hi);
    bool ok = true;
    int t = 0, oi = 0, slot = 0, round = 0;
    int lens = 0;
    for (int pair = lo; pair < hi && ok; ++pair) {
      const int n = pair - lo;
      if ((n & 31) == 0) lens = pair_lens(p, pair, hi, lane);
      const int len = __shfl_sync(0xffffffffu, lens, n & 31);
      const int nt = (len + kBN - 1) / kBN;
      if (nt == 0) continue;
      const uint32_t d_tmem = tmem + 2 * kN + (oi & 1) * C::kOCols;
      for (int j = 0; j < nt && ok; ++j) {
        // P_t written (so S_t, and with it this slot's K and V, had landed)
        ok = __all_sync(0xffffffffu, mbar_wait(&sh->p_full[t & 1], (t >> 1) & 1, abort_flag));
        // the pair's first product overwrites O: its epilogue two pairs back is done
        if (ok && j == 0)
          ok = __all_sync(0xffffffffu,
                          mbar_wait(&sh->o_free[oi & 1], ((oi >> 1) & 1) ^ 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          // A = V^T: 16 key rows per step (8-row groups 1024 B apart)
          const uint64_t da0 = smem_desc_sw128(
              smem_addr(ring + slot * C::kSlotBytes + C::kTileBytes), C::kVLbo, 1024);
          // B = P: 16 keys = 32 bytes of each 128-byte row
          const uint64_t db0 = smem_desc_sw128(smem_addr(pbuf + (t & 1) * C::kPBytes), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < C::kPvSteps; ++kk) {
            // d = 64: P rows 0..31 (both halves) per step; d = 128: 16 rows,
            // the second 64 keys kQBlk further
            const uint32_t pb = D == 64 ? kk * 32 : (kk >> 2) * C::kQBlk + (kk & 3) * 32;
            tc_mma_ss(d_tmem, da0 + ((kk * 16 * 128) >> 4), db0 + (pb >> 4), idesc_o,
                      (j > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&sh->pv_done[t & 1]);
          tc_commit(&sh->kv_empty[slot]);
        }
        __syncwarp();
        last_commit = &sh->kv_empty[slot];
        last_parity = round & 1;
        ++t;
        if (++slot == C::kSlots) {
          slot = 0;
          ++round;
        }
      }
      ++oi;
    }
  } else {
    // ---- softmax and epilogue: thread k = key k of a tile / TMEM lane k ----
    const int k = threadIdx.x;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    // O^T lanes: d = 128, value dim k; d = 64, value dim k % 64 of the first
    // (warps 0-1) or second (warps 2-3) key half's partial output
    const int o_col = D == 64 && warp >= 2 ? kN : 0;
    const int vdim = D == 64 ? (k & 63) : k;
    const bool stores = D == 128 || warp < 2;  // threads that write output
    griddep_wait();
    int lo, hi;
    pair_range(p, lane, lo, hi);
    bool ok = true;
    int t = 0, oi = 0;
    int lens = 0;
    for (int pair = lo; pair < hi; ++pair) {
      const int n = pair - lo;
      if ((n & 31) == 0) lens = pair_lens(p, pair, hi, lane);
      const int len = __shfl_sync(0xffffffffu, lens, n & 31);
      const int nt = (len + kBN - 1) / kBN;
      const int b = pair / p.Hkv, g = pair - b * p.Hkv;
      // element (row r, value dim vdim) of this pair's output
      auto out_at = [&](int r) -> uint16_t * {
        const int hl = r / p.Lq, pos = r - hl * p.Lq;
        const int h = g * group + hl;
        const size_t row = p.layout == kLayoutBHSD
                               ? (static_cast<size_t>(b) * p.H + h) * p.Lq + pos
                               : (static_cast<size_t>(b) * p.Lq + pos) * p.H + h;
        return out + row * D + vdim;
      };
      // statistics row of row r (the [B, H, Lq] lse)
      auto lse_at = [&](int r) -> float * {
        const int hl = r / p.Lq, pos = r - hl * p.Lq;
        return p.lse + (static_cast<size_t>(b) * p.H + g * group + hl) * p.Lq + pos;
      };
      if (nt == 0) {
        // no key at all: the rows are +0.0
        if (stores)
          for (int r = 0; r < R; ++r) *out_at(r) = 0;
        if (p.lse != nullptr && k == 0)
          for (int r = 0; r < R; ++r) *lse_at(r) = INFINITY;
        continue;
      }
      // keys j < jbase (+ the row's position under the cached-decoding mask)
      const int jbase = tail ? len - p.Lq + 1 : len;
      float m[RP], l[RP];
#pragma unroll
      for (int r = 0; r < RP; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
      }
      for (int j = 0; j < nt; ++j) {
        const bool okw =
            __all_sync(0xffffffffu, mbar_wait(&sh->s_full[t & 1], (t >> 1) & 1, abort_flag));
        float x[RP];
        if (okw) {
          tc_fence_after();
          uint32_t s[RP];
          tmem_ld_cols(tmem + lane_base + (t & 1) * kN, s);
          tmem_wait_ld();
#pragma unroll
          for (int r = 0; r < RP; ++r) {
            x[r] = __uint_as_float(s[r]) * p.scale_log2;
            if (RP > 1 && r >= R) x[r] = -INFINITY;  // padding rows of the product
          }
          if (j * kBN + kBN > jbase) {  // a tile that crosses some row's limit
            const int key = j * kBN + k;
            int pos = 0;
#pragma unroll
            for (int r = 0; r < RP; ++r) {
              if (key >= jbase + (tail ? pos : 0)) x[r] = -INFINITY;
              if (++pos == p.Lq) pos = 0;
            }
          }
#pragma unroll
          for (int r = 0; r < RP; ++r) {
            const float v = warp_max(x[r]);
            if (lane == 0) sh->red[t & 1][warp][r] = v;
          }
        }
        ok = named_barrier_and(kBarSoftmax, kSoftmaxThreads, ok && okw);
        if (!ok) break;
        // the lazy running maximum (identical in every thread)
        float alpha[RP];
        bool rescale = false;
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          const float tm = fmaxf(fmaxf(sh->red[t & 1][0][r], sh->red[t & 1][1][r]),
                                 fmaxf(sh->red[t & 1][2][r], sh->red[t & 1][3][r]));
          const bool up = tm > m[r] + kRescaleThreshold;
          const bool moved = up && m[r] != -INFINITY;
          alpha[r] = moved ? ex2_approx(m[r] - tm) : 1.f;
          l[r] *= alpha[r];
          rescale |= moved;
          m[r] = up ? tm : m[r];
        }
        if (rescale) {
          // O holds PV products of earlier tiles of this pair: wait for the
          // last one (PV_{t-1}), then scale its columns
          const int u = t - 1;
          const bool okr = __all_sync(
              0xffffffffu, mbar_wait(&sh->pv_done[u & 1], (u >> 1) & 1, abort_flag));
          if (okr) {
            tc_fence_after();
            uint32_t o[RP];
            const uint32_t ta = tmem + lane_base + 2 * kN + (oi & 1) * C::kOCols + o_col;
            tmem_ld_cols(ta, o);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < RP; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha[c]);
            tmem_st_cols(ta, o);
            tmem_wait_st();
          }
          ok = okr;
        }
        // P buffer t % 2 held P_{t-2}: its product must be done reading it
        if (t >= 2 && ok)
          ok = __all_sync(0xffffffffu,
                          mbar_wait(&sh->pv_done[t & 1], ((t - 2) >> 1) & 1, abort_flag));
        // row r of P_t: keys of this tile, bf16, 128B-swizzled rows; the
        // second 64 keys in the second 2 KB (rows 16..31 of the d = 64 product)
        const uint32_t pb = smem_addr(pbuf + (t & 1) * C::kPBytes) + (k >> 6) * C::kQBlk;
        const uint32_t kc = static_cast<uint32_t>(k & 63);
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          const float pr = ex2_approx(x[r] - (m[r] == -INFINITY ? 0.f : m[r]));
          l[r] += pr;
          st_shared_u16(pb + r * 128 + (((kc >> 3) ^ (r & 7)) << 4) + (kc & 7) * 2,
                        bf16_bits(pr));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&sh->p_full[t & 1]);
        ++t;
      }
      if (!ok) break;
      // ---- epilogue: l = sum over the key slots, O = O^T / l -------------
#pragma unroll
      for (int r = 0; r < RP; ++r) {
        const float v = warp_sum(l[r]);
        if (lane == 0) sh->lsum[warp][r] = v;
      }
      const int u = t - 1;
      const bool oke =
          __all_sync(0xffffffffu, mbar_wait(&sh->pv_done[u & 1], (u >> 1) & 1, abort_flag));
      uint32_t o[RP];
      if (oke) {
        tc_fence_after();
        tmem_ld_cols(tmem + lane_base + 2 * kN + (oi & 1) * C::kOCols + o_col, o);
        tmem_wait_ld();
        if (D == 64 && warp >= 2) {
#pragma unroll
          for (int r = 0; r < RP; ++r) sh->xo[r][vdim] = __uint_as_float(o[r]);
        }
      }
      tc_fence_before();
      mbar_arrive(&sh->o_free[oi & 1]);
      ++oi;
      ok = named_barrier_and(kBarSoftmax, kSoftmaxThreads, ok && oke);
      if (!ok) break;
      if (stores) {
#pragma unroll
        for (int r = 0; r < RP; ++r)
          if (r < R) {
            const float lt = (sh->lsum[0][r] + sh->lsum[1][r]) + (sh->lsum[2][r] + sh->lsum[3][r]);
            float acc = __uint_as_float(o[r]);
            if (D == 64) acc += sh->xo[r][vdim];
            // a row with no allowed key is stored as +0.0
            *out_at(r) = bf16_bits(lt > 0.f ? acc * (1.f / lt) : 0.f);
            if (p.lse != nullptr && k == 0) *lse_at(r) = lt > 0.f ? m[r] + __log2f(lt) : INFINITY;
          }
      }
      // lsum and xo are rewritten only after the next pair's first tile
      // barrier, which every thread reaches after the reads above
    }
  }

  // ---- teardown --------------------------------------------------------------
  if (*abort_flag && warp == 4 && lane == 0) {
    for (int idx = issued - C::kSlots; idx < issued; ++idx)
      if (idx >= 0) (void)wait_teardown(&sh->kv_full[idx % C::kSlots], (idx / C::kSlots) & 1);
    for (int qi = q_issued - 2; qi < q_issued; ++qi)
      if (qi >= 0) (void)wait_teardown(&sh->q_full[qi & 1], (qi >> 1) & 1);
  }
  if (*abort_flag && (warp == 5 || warp == 6) && lane == 0 && last_commit != nullptr)
    (void)wait_teardown(last_commit, last_parity);
  if (*abort_flag && threadIdx.x == 0) atomicExch(p.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

template <int D, int RP>
cudaError_t launch_decode_impl(const DecodeMaps &maps, const Problem &p, void *out, int num_sms,
                               cudaStream_t stream) {
  static_assert(smem_bytes<D>() <= 232448, "shared memory budget");
  static_assert(Cfg<D>::kSlots <= kMaxSlots, "ring size");
  constexpr size_t kSmem = smem_bytes<D>();
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(attn_decode_tc_kernel<D, RP>), static_cast<int>(kSmem));
  if (e != cudaSuccess) return e;
  const long long npairs = static_cast<long long>(p.B) * p.Hkv;
  if (npairs <= 0) return cudaSuccess;
  const int grid = static_cast<int>(npairs < num_sms ? npairs : num_sms);
  // programmatic dependent launch: set-up may overlap the previous kernel's
  // tail; every role waits for it before its first global memory access
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_decode_tc_kernel<D, RP>, maps, p,
                            static_cast<uint16_t *>(out));
}

template <int D>
cudaError_t launch_decode_rows(const DecodeMaps &maps, const Problem &p, void *out, int num_sms,
                               cudaStream_t stream) {
  const int R = (p.H / p.Hkv) * p.Lq;
  if (R <= 1) return launch_decode_impl<D, 1>(maps, p, out, num_sms, stream);
  if (R <= 2) return launch_decode_impl<D, 2>(maps, p, out, num_sms, stream);
  if (R <= 4) return launch_decode_impl<D, 4>(maps, p, out, num_sms, stream);
  if (R <= 8) return launch_decode_impl<D, 8>(maps, p, out, num_sms, stream);
  return launch_decode_impl<D, 16>(maps, p, out, num_sms, stream);
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeMaps &maps, const Problem &p, void *out, int num_sms,
                             cudaStream_t stream) {
  if (p.Hkv <= 0 || (p.H / p.Hkv) * p.Lq > kN) return cudaErrorInvalidValue;
  if (p.dk == 128) return launch_decode_rows<128>(maps, p, out, num_sms, stream);
  return launch_decode_rows<64>(maps, p, out, num_sms, stream);
}

}  // namespace mha
