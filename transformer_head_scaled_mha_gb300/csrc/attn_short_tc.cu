// Packed short-sequence attention on the tcgen05 tensor cores (bf16, d = 64).
//
// Sentence-length attention (Lq, Lk <= 128) is bound by HBM traffic, not by
// arithmetic: each (batch, head) pair is one small Q K^T and one small P V.
// This kernel packs P = 128 / max(Rq, Rk) pairs into one 128-row tile (Rq,
// Rk: Lq, Lk rounded up to powers of two) so one tcgen05.mma covers all of
// them; products between different pairs land in off-diagonal blocks that are
// never read.  A unit holds P consecutive heads of one batch element; with
// shared key/value heads (grouped- or multi-query attention) pair h reads the
// K and V of head h / (H / H_kv).  Each CTA is persistent (one per SM) and
// walks the units u = blockIdx.x, + gridDim.x, ...
//
// Warp roles (384 threads):
//   warps 0-3, 4-7  two softmax warpgroups; unit n goes to warpgroup n % 2,
//                   thread t owns tile row t
//   warp  8         TMA producer: Q, K, V of a unit into a 4-stage ring
//   warp  9         TMEM owner and MMA issuer
//   warps 10-11     idle; they complete the third warpgroup so its register
//                   budget can be handed to the softmax warpgroups
// Per unit (the four steps of scaled dot-product attention):
//   S = Q K^T              tcgen05.mma -> TMEM (fp32), one region per warpgroup
//   mask, scale, softmax   tcgen05.ld of the 32-column chunks the warp's rows
//                          can use -> registers; exp2 against the row max
//   P (bf16) -> TMEM       the warpgroup's own P columns, so S of its next
//                          unit is computed while P V still reads P
//   O = P V                tcgen05.mma (A = P from TMEM) -> TMEM
//   O / rowsum -> bf16     tcgen05.ld; each warp stages its 32 rows in a
//                          swizzled 4 KiB buffer and writes them back with
//                          stores that each cover four whole rows
// The MMA warp issues S for unit n + 2 as soon as the warpgroup posted P for
// unit n, and P V for unit n once the warpgroup has read O of unit n - 2.
// Padded sequences load only their first ceil(len/8)*8 rows, as one TMA box
// of that height per tensor and pair, so padding costs no HBM reads (a CTA's
// first unit loads whole tiles instead, so it does not wait for the lengths).
// Masked keys get exactly zero weight; padded query rows and rows without any
// allowed key are stored as +0.  All tensor maps are 4-D (d, L, heads, B), so
// the [B, H, L, d] and [B, L, H, d] layouts run the same code.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kD = 64;
constexpr int kStages = 4;
constexpr int kTileRows = 128;
constexpr int kTileBytes = kTileRows * kD * 2;  // 16 KiB per operand tile
constexpr int kStageBytes = 3 * kTileBytes;     // Q | K | V
constexpr int kThreads = 384;  // 3 warpgroups
constexpr int kWgThreads = 128;
// Register split: launched at 168 per thread (384 x 168 = 64512); the control
// warpgroup drops to 80 and the softmax warpgroups rise to 208 (no spills).
constexpr uint32_t kRegsSoftmax = 208;
constexpr uint32_t kRegsControl = 80;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsControl <= kThreads * 168, "register split");
constexpr uint32_t kTmemCols = 512;
// TMEM columns of warpgroup w: S (fp32) [128 w, +128), P (bf16 pairs)
// [256 + 64 w, +64), O (fp32) [384 + 64 w, +64).  P has its own columns so
// the next S of a warpgroup can be computed while P V still reads P.
constexpr uint32_t kSCol0 = 0;
constexpr uint32_t kPCol0 = 256;
constexpr uint32_t kOCol0 = 384;

struct __align__(8) Barriers {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t s_full[2];   // S of the warpgroup's unit is in TMEM
  uint64_t p_full[2];   // the warpgroup read its S and wrote P
  uint64_t pv_done[2];  // P V done: O ready, P columns free
  uint64_t o_free[2];   // the warpgroup read O
  uint32_t tmem_base;
  int abort_flag;
};

constexpr int kStagingBytes = 32 * 128;  // one warp's 32 output rows
constexpr size_t kSmemBytes = 1024 /* alignment slack */ + kStages * kStageBytes +
                              8 * kStagingBytes + sizeof(Barriers);

__device__ __forceinline__ int clamp_len(const Problem &p, int b) {
  if (!(p.mask & (kMaskKeyPadding | kMaskQueryPadding))) return p.Lk;
  const int l = p.key_lengths[b];
  return l < 0 ? 0 : (l > p.Lk ? p.Lk : l);
}

// (batch element, head group) of the units u0, u0 + step, u0 + 2 step, ...,
// stepped without a division per unit
struct UnitWalk {
  int b, hu, db, dh, per_b;
  __device__ __forceinline__ UnitWalk(int u0, int step, int per_b_)
      : b(u0 / per_b_), hu(u0 % per_b_), db(step / per_b_), dh(step % per_b_), per_b(per_b_) {}
  __device__ __forceinline__ void next() {
    b += db;
    hu += dh;
    if (hu >= per_b) {
      hu -= per_b;
      ++b;
    }
  }
};

__device__ __forceinline__ bool wait_teardown(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity))
    if (global_timer_ns() - t0 > 100000000ull) return false;
  return true;
}

// Rows [0, rows) of one pair (rounded up to a multiple of 8) as one TMA box
// of exactly that height: each box costs the TMA unit a fixed overhead, so
// one box per pair and tensor beats a split into power-of-two pieces.
__device__ __forceinline__ uint32_t box_bytes(int rows) {
  return static_cast<uint32_t>((rows + 7) / 8) * 1024u;
}
__device__ __forceinline__ void load_rows(uint8_t *dst, const CUtensorMap *maps, uint64_t *bar,
                                          int rows, int head, int b) {
  const int n8 = (rows + 7) / 8;
  if (n8 > 0) tma_load_4d(dst, &maps[n8 - 1], bar, 0, 0, head, b);
}

// One 32-column chunk of a row's scores (raw fp32 bits), sign-flipped by
// `sgn` (a negative scale is applied as |scale| to -s), with columns outside
// lo <= c < hi set to -inf when `mask`.  Both steps are skipped when they do
// nothing (the usual case), which keeps the executed code small.
__device__ __forceinline__ void chunk_prepare(uint32_t (&v)[32], int c0, uint32_t sgn, bool mask,
                                              int lo, int hi) {
  if (sgn) {
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] ^= sgn;
  }
  if (mask) {
    // bit e set: column c0 + e is kept
    const int a = min(max(lo - c0, 0), 32), z = min(max(hi - c0, 0), 32);
    const uint32_t upto_z = z >= 32 ? 0xffffffffu : (1u << z) - 1u;
    const uint32_t upto_a = a >= 32 ? 0xffffffffu : (1u << a) - 1u;
    const uint32_t keep = upto_z & ~upto_a;
#pragma unroll
    for (int e = 0; e < 32; ++e)
      if (!((keep >> e) & 1u)) v[e] = __float_as_uint(-INFINITY);
  }
}
__device__ __forceinline__ float chunk_max(const uint32_t (&v)[32]) {
  float t[11];
#pragma unroll
  for (int k = 0; k < 10; ++k)
    t[k] = fmax3(__uint_as_float(v[3 * k]), __uint_as_float(v[3 * k + 1]),
                 __uint_as_float(v[3 * k + 2]));
  t[10] = fmaxf(__uint_as_float(v[30]), __uint_as_float(v[31]));
  return fmax3(fmax3(t[0], t[1], t[2]), fmax3(t[3], t[4], t[5]),
               fmax3(fmax3(t[6], t[7], t[8]), t[9], t[10]));
}
// Multiplies the 32 bf16 P values of one chunk (16 TMEM columns) by f.
__device__ __noinline__ void rescale_p(uint32_t taddr, float f) {
  uint32_t r[16];
  tmem_ld16(taddr, r);
  tmem_wait_ld();
#pragma unroll
  for (int t = 0; t < 16; ++t)
    r[t] = pack_bf16x2(__uint_as_float(r[t] << 16) * f, __uint_as_float(r[t] & 0xffff0000u) * f);
  tmem_st16(taddr, r);
  tmem_wait_st();
}

// p_c = exp2(s_c * sl - m) for one chunk, packed into 16 bf16x2 columns;
// returns the chunk's sum of p (fp32)
__device__ __forceinline__ float chunk_exp_pack(const uint32_t (&v)[32], float sl, float m,
                                                uint32_t (&pk)[16]) {
  const uint64_t sc = f2_pack(sl, sl);
  const uint64_t nm = f2_pack(-m, -m);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float a, b;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sc, nm), a, b);
    a = ex2_approx(a);
    b = ex2_approx(b);
    acc[(e >> 1) & 3] = f2_add(acc[(e >> 1) & 3], f2_pack(a, b));
    pk[e >> 1] = pack_bf16x2(a, b);
  }
  acc[0] = f2_add(acc[0], acc[1]);
  acc[2] = f2_add(acc[2], acc[3]);
  acc[0] = f2_add(acc[0], acc[2]);
  float lo, hi;
  f2_unpack(acc[0], lo, hi);
  return lo + hi;
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_short_tc_kernel(const __grid_constant__ ShortMaps maps, const ShortGeom g,
                         const Problem p, void *out) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *stage_base = smem;
  uint8_t *staging = smem + kStages * kStageBytes;  // 8 softmax warps x 4 KiB
  Barriers *bars = reinterpret_cast<Barriers *>(staging + 8 * kStagingBytes);
  volatile int *abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int group = p.H / p.Hkv;  // query heads per key/value head
  // Causal 128-row tiles: row 96 + t needs four 32-key chunks of softmax,
  // row t one, and TMEM lanes 32 q .. 32 q + 31 belong to the warps on SM
  // sub-partition q.  Warpgroup 1 therefore holds its query rows with the
  // 32-row blocks in reverse order, so each sub-partition gets one heavy and
  // one light warp.
  const bool rev = (p.mask & kMaskCausal) && g.Rq == 128 && !g.rows_q;
  const int n_local = (static_cast<int>(blockIdx.x) < g.units)
                          ? (g.units - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1
                          : 0;

  // ---- setup -------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&bars->s_full[w], 1);
      mbar_init(&bars->p_full[w], kWgThreads);
      mbar_init(&bars->pv_done[w], 1);
      mbar_init(&bars->o_free[w], kWgThreads);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&maps.q_full);
    tma_prefetch_desc(group == 1 ? &maps.k_full : &maps.k_one);
    tma_prefetch_desc(group == 1 ? &maps.v_full : &maps.v_one);
    // While the previous grid drains, warm L2 with this CTA's first two
    // units (whole tiles) and first three lengths.  All global writes land
    // in L2, so an L2 prefetch can never make a later read stale; the reads
    // that count still come after the dependency wait below.
    for (int n = 0; n < 3 && n < n_local; ++n) {
      const int u = blockIdx.x + n * gridDim.x;
      const int b = u / g.units_per_b, h0 = (u % g.units_per_b) * g.P;
      if (p.key_lengths != nullptr) prefetch_l2(p.key_lengths + b);
      if (n < 2) {
        tma_prefetch_l2_4d(&maps.q_full, 0, 0, h0, b);
        if (group == 1) {
          tma_prefetch_l2_4d(&maps.k_full, 0, 0, h0, b);
          tma_prefetch_l2_4d(&maps.v_full, 0, 0, h0, b);
        }
      }
    }
  }
  if (warp == 9) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // V rows that a padded unit does not load keep earlier contents; start
  // from zeros so they are always finite (their weights are exactly zero, and
  // 0 * NaN would not be).  Unloaded K and Q rows are masked by selection.
  if (g.rows_k) {
    for (int i = threadIdx.x; i < kStages * kTileBytes / 16; i += kThreads) {
      const int st = i / (kTileBytes / 16), off = i % (kTileBytes / 16);
      reinterpret_cast<uint4 *>(stage_base + st * kStageBytes + 2 * kTileBytes)[off] =
          make_uint4(0, 0, 0, 0);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // Everything above overlaps the previous launch's tail when launched as a
  // programmatic dependent; global memory is touched only after this wait.
  griddep_wait();
  griddep_launch_dependents();

  int issued = 0;                   // producer: units whose loads were issued
  uint64_t *last_commit = nullptr;  // MMA issuer: barrier of the last commit
  uint32_t last_commit_parity = 0;
  if (warp >= 8) {
   regs_dec<kRegsControl>();
   if (warp == 8) {
    // ---- TMA producer (lane pp handles pair pp of the unit) -----------------
    const int pp = lane;
    const bool need_len = g.rows_q || g.rows_k;
    // lane pp's pair length for the unit at `at` (unit n), read two units
    // ahead of its use
    auto len_at = [&](const UnitWalk &at, int n) -> int {
      return (need_len && n < n_local && pp < g.P && at.hu * g.P + pp < p.H) ? clamp_len(p, at.b)
                                                                           : 0;
    };
    UnitWalk cur(blockIdx.x, gridDim.x, g.units_per_b);
    UnitWalk ahead(blockIdx.x + gridDim.x, gridDim.x, g.units_per_b);
    int len_n1 = len_at(ahead, 1);
    ahead.next();
    int len_n2 = len_at(ahead, 2);
    for (int n = 0; n < n_local; ++n, cur.next()) {
      const int s = n % kStages;
      const int b = cur.b, h0 = cur.hu * g.P;
      // key/value head of pair pp (a pair past the last head, whose rows are
      // never stored, reads the last head so every box is in bounds)
      const int hq = min(h0 + pp, p.H - 1);
      const int hkv = group == 1 ? hq : hq / group;
      // the first unit loads whole tiles: no wait for the lengths
      const bool rows_q = g.rows_q && n > 0, rows_k = g.rows_k && n > 0;
      const bool has_pair = pp < g.P && h0 + pp < p.H;
      const int len = n > 0 ? len_n1 : 0;
      if (n > 0) {
        ahead.next();
        len_n1 = len_n2;
        len_n2 = len_at(ahead, n + 2);
      }
      uint32_t bytes = 0;
      if (has_pair && rows_q) bytes += box_bytes(min(len, p.Lq));
      if (has_pair && rows_k) bytes += 2 * box_bytes(len);
      bytes = __reduce_add_sync(0xffffffffu, bytes);
      if (!rows_q) bytes += g.P * g.Rq * 128;
      if (!rows_k) bytes += 2 * g.P * g.Rk * 128;
      if (!mbar_wait(&bars->empty[s], ((n / kStages) & 1) ^ 1, abort_flag)) break;
      uint8_t *sq = stage_base + s * kStageBytes;
      uint8_t *sk = sq + kTileBytes;
      uint8_t *sv = sk + kTileBytes;
      if (lane == 0) mbar_arrive_expect_tx(&bars->full[s], bytes);
      __syncwarp();
      // whole tiles: one box of P heads, or with shared key/value heads one
      // box per pair (heads past H read as zeros and are never stored)
      if (rev && (n & 1)) {
        // warpgroup 1 of a causal tile: reversed 32-row blocks (see above)
        if (lane < 4)
          tma_load_4d(sq + lane * 32 * 128, &maps.q_blk32, &bars->full[s], 0, (3 - lane) * 32, h0,
                      b);
      } else if (lane == 0 && !rows_q) {
        tma_load_4d(sq, &maps.q_full, &bars->full[s], 0, 0, h0, b);
      }
      if (lane == 0) {
        if (!rows_k && group == 1) {
          tma_load_4d(sk, &maps.k_full, &bars->full[s], 0, 0, h0, b);
          tma_load_4d(sv, &maps.v_full, &bars->full[s], 0, 0, h0, b);
        }
      }
      if (!rows_k && group != 1 && pp < g.P) {
        tma_load_4d(sk + pp * g.Rk * 128, &maps.k_one, &bars->full[s], 0, 0, hkv, b);
        tma_load_4d(sv + pp * g.Rk * 128, &maps.v_one, &bars->full[s], 0, 0, hkv, b);
      }
      if (has_pair && rows_q) load_rows(sq + pp * g.Rq * 128, maps.q_rows, &bars->full[s],
                                        min(len, p.Lq), h0 + pp, b);
      if (has_pair && rows_k) {
        load_rows(sk + pp * g.Rk * 128, maps.k_rows, &bars->full[s], len, hkv, b);
        load_rows(sv + pp * g.Rk * 128, maps.v_rows, &bars->full[s], len, hkv, b);
      }
      __syncwarp();
      issued = n + 1;
    }
  } else if (warp == 9) {
    // ---- MMA issuer (lane 0) ----------------------------------------------
    const uint32_t n_keys = static_cast<uint32_t>(g.P * g.Rk);  // multiple of 16, <= 128
    const uint32_t idesc_s = idesc_bf16_f32(128, n_keys, 0);
    const uint32_t idesc_o = idesc_bf16_f32(128, kD, 1);
    // Fixed order S_0, S_1, then for each unit n: S for n + 2 (warpgroup
    // n % 2 is done reading S_n once it posted P_n), then P V for n (its O
    // columns are free once the warpgroup read O of unit n - 2).  Every wait
    // suspends in hardware until its phase completes.
    auto issue_s = [&](int ns) -> bool {
      const int s = ns % kStages, w = ns & 1;
      if (!mbar_wait(&bars->full[s], (ns / kStages) & 1, abort_flag)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t sq = smem_addr(stage_base + s * kStageBytes);
        const uint32_t sk = sq + kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          tc_mma_ss(tmem + kSCol0 + w * 128, smem_desc_sw128(sq + kk * 32, 16, 1024),
                    smem_desc_sw128(sk + kk * 32, 16, 1024), idesc_s, kk > 0);
        tc_commit(&bars->s_full[w]);
      }
      __syncwarp();
      last_commit = &bars->s_full[w];
      last_commit_parity = (ns >> 1) & 1;
      return true;
    };
    bool ok = true;
    for (int ns = 0; ok && ns < 2 && ns < n_local; ++ns) ok = issue_s(ns);
    for (int n = 0; ok && n < n_local; ++n) {
      const int s = n % kStages, w = n & 1;
      if (!mbar_wait(&bars->p_full[w], (n >> 1) & 1, abort_flag)) break;
      if (n + 2 < n_local && !(ok = issue_s(n + 2))) break;
      if (n >= 2 && !mbar_wait(&bars->o_free[w], ((n - 2) >> 1) & 1, abort_flag)) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t sv = smem_addr(stage_base + s * kStageBytes + 2 * kTileBytes);
        for (uint32_t kk = 0; kk < n_keys / 16; ++kk)
          // A = P (TMEM, 16 keys = 8 columns per step); B = V (MN-major)
          tc_mma_ts(tmem + kOCol0 + w * kD, tmem + kPCol0 + w * 64 + kk * 8,
                    smem_desc_sw128(sv + kk * 16 * 128, 1024, 1024), idesc_o, kk > 0);
        tc_commit(&bars->pv_done[w]);
        tc_commit(&bars->empty[s]);
      }
      __syncwarp();
      last_commit = &bars->empty[s];
      last_commit_parity = (n / kStages) & 1;
    }
   }
  } else {
    regs_inc<kRegsSoftmax>();
    // ---- softmax + epilogue: warpgroup w takes units n = w, w + 2, ... -----
    const int w = warp >> 2;
    const int r = threadIdx.x & 127;  // tile row = TMEM lane
    const bool my_rev = rev && w == 1;  // query row of tile row r
    const int pr = r / g.Rq, i = my_rev ? ((3 - (r >> 5)) << 5) | (r & 31) : r % g.Rq;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_tmem = tmem + lane_base + kSCol0 + w * 128;
    const uint32_t p_tmem = tmem + lane_base + kPCol0 + w * 64;
    const uint32_t o_tmem = tmem + lane_base + kOCol0 + w * kD;
    // output rows: this lane stores 16-byte piece (lane & 7) of warp rows
    // 4 t + (lane >> 3), t = 0..7, so each store instruction writes four
    // whole 128-byte rows
    const int rq_shift = __ffs(g.Rq) - 1;
    const long long row_stride = p.layout == kLayoutBHSD ? 128 : 128LL * p.H;
    const long long head_stride = p.layout == kLayoutBHSD ? 128LL * p.Lq : 128;
    const long long batch_stride = 128LL * p.Lq * p.H;
    // a negative scale is applied as |scale| to sign-flipped scores
    const uint32_t sgn = p.scale_log2 < 0.f ? 0x80000000u : 0u;
    const float sl = fabsf(p.scale_log2);

    // this thread's row is real in the unit at `at`
    auto row_valid = [&](const UnitWalk &at) -> bool {
      return pr < g.P && at.hu * g.P + pr < p.H && i < p.Lq;
    };
    UnitWalk cur(blockIdx.x + w * gridDim.x, 2 * gridDim.x, g.units_per_b);
    UnitWalk nxt = cur;
    nxt.next();
    int len_cur = (w < n_local && row_valid(cur)) ? clamp_len(p, cur.b) : 0;
    float rowsum_prev = 0.f;  // row sum of the unit whose epilogue is pending
    bool pending_zero = true;
    int prev_b = 0, prev_h0 = 0;  // the pending unit's batch element and first head
    for (int n = w; n < n_local + 2; n += 2, cur.next(), nxt.next()) {
      float rowsum = 0.f;
      bool zero_row = true;
      // load ahead of its use
      const int len_next = (n + 2 < n_local && row_valid(nxt)) ? clamp_len(p, nxt.b) : 0;
      if (n < n_local) {
        const int k = n >> 1;  // this warpgroup's k-th unit
        const bool valid = row_valid(cur);
        const int len = len_cur;
        int jmax = p.Lk;
        if (p.mask & kMaskKeyPadding) jmax = min(jmax, len);
        if (p.mask & kMaskCausal) jmax = min(jmax, i + 1);
        const bool qpad = (p.mask & kMaskQueryPadding) && i >= len;
        if (!valid || qpad) jmax = 0;
        const int col_lo = pr * g.Rk;
        // 32-column chunks any row of this warp can use
        const unsigned lo = __reduce_min_sync(0xffffffffu, jmax > 0 ? col_lo : 1 << 20);
        const unsigned hi = __reduce_max_sync(0xffffffffu, jmax > 0 ? col_lo + jmax : 0);
        const int ch_lo = hi > 0 ? static_cast<int>(lo / 32) : 4;
        const int ch_hi = hi > 0 ? static_cast<int>((hi + 31) / 32) : 0;

        if (!mbar_wait(&bars->s_full[w], k & 1, abort_flag)) break;
        tc_fence_after();
        // keep only this row's keys [col_lo, col_lo + jmax).  One pass over
        // the chunks: exponents are taken against the first chunk's max m;
        // a later chunk may exceed m by up to 2^8 (P stays far from bf16
        // overflow, and numerator and denominator share m, so the quotient
        // is unchanged).  A row whose max grows further rescales the P it
        // already wrote (rare: the scores would have to climb steeply along
        // the keys).
        const int lo_c = col_lo, hi_c = col_lo + jmax;
        float ms = -INFINITY;  // reference max, scaled (log2 units)
        bool gave_up = false;
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t pk[16];
          if (ch >= ch_lo && ch < ch_hi) {
            uint32_t v[32];
            tmem_ld32(s_tmem + ch * 32, v);
            tmem_wait_ld();
            const bool mask = __any_sync(0xffffffffu, ch * 32 < lo_c || ch * 32 + 32 > hi_c);
            chunk_prepare(v, ch * 32, sgn, mask, lo_c, hi_c);
            const float cm = chunk_max(v) * sl;  // -inf when no key of the chunk is kept
            if (ms == -INFINITY) ms = cm;
            const bool climb = cm > ms + 8.f;
            if (__any_sync(0xffffffffu, climb)) {
              const float f = climb ? ex2_approx(ms - cm) : 1.f;
              rowsum *= f;
              for (int c = ch_lo; c < ch; ++c) rescale_p(p_tmem + c * 16, f);
              if (climb) ms = cm;
            }
            const float cs = chunk_exp_pack(v, sl, ms == -INFINITY ? 0.f : ms, pk);
            rowsum += cs;
          } else {
#pragma unroll
            for (int t = 0; t < 16; ++t) pk[t] = 0u;
          }
          // the P columns are free once P V of this warpgroup's previous unit ran
          if (ch == 0 && k > 0 && !mbar_wait(&bars->pv_done[w], (k - 1) & 1, abort_flag)) {
            gave_up = true;
            break;
          }
          if (ch == 0) tc_fence_after();
          tmem_st16(p_tmem + ch * 16, pk);
        }
        if (gave_up) break;
        zero_row = ms == -INFINITY;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[w]);
      }
      // epilogue of this warpgroup's previous unit (its P V ran meanwhile)
      if (n - 2 >= 0 && n - 2 < n_local) {
        const int pn = n - 2;
        if (!mbar_wait(&bars->pv_done[w], (pn >> 1) & 1, abort_flag)) break;
        tc_fence_after();
        uint32_t o[2][32];
        tmem_ld32(o_tmem, o[0]);
        tmem_ld32(o_tmem + 32, o[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars->o_free[w]);
        // bf16 row into this warp's staging rows (128-byte swizzle), then
        // read back row-major so every store covers four whole rows
        const float inv = pending_zero ? 0.f : 1.f / rowsum_prev;
        uint8_t *stg = staging + warp * kStagingBytes;
        const uint32_t so = smem_addr(stg);
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          uint32_t wv[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int c = c8 * 8 + 2 * t;
            wv[t] = pending_zero ? 0u
                                 : pack_bf16x2(__uint_as_float(o[c >> 5][c & 31]) * inv,
                                               __uint_as_float(o[c >> 5][(c + 1) & 31]) * inv);
          }
          st_shared_v4(so + sw128_offset(lane, c8), wv[0], wv[1], wv[2], wv[3]);
        }
        __syncwarp();
        const int b = prev_b, h0 = prev_h0;
        uint8_t *obase = static_cast<uint8_t *>(out) + b * batch_stride;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int rr = 4 * t + (lane >> 3);           // warp row
          const int row = (warp & 3) * 32 + rr;          // tile row
          const int pr_o = row >> rq_shift;
          const int i_o = my_rev ? ((3 - (row >> 5)) << 5) | (row & 31) : row & (g.Rq - 1);
          const uint4 val = ld_shared_v4(so + sw128_offset(rr, lane & 7));
          if (pr_o < g.P && h0 + pr_o < p.H && i_o < p.Lq)
            st_global_v4(obase + (h0 + pr_o) * head_stride + i_o * row_stride + (lane & 7) * 16,
                         val);
        }
        __syncwarp();
      }
      rowsum_prev = rowsum;
      pending_zero = zero_row;
      len_cur = len_next;
      prev_b = cur.b;
      prev_h0 = cur.hu * g.P;
    }
  }

  // ---- teardown ------------------------------------------------------------
  if (*abort_flag && warp == 8 && lane == 0) {
    // let copies already in flight land before the CTA's shared memory goes away
    for (int n = issued - kStages; n < issued; ++n)
      if (n >= 0) (void)wait_teardown(&bars->full[n % kStages], (n / kStages) & 1);
  }
  if (*abort_flag && warp == 9 && lane == 0 && last_commit != nullptr) {
    // tcgen05 ops complete in order: the last commit covers all of them
    (void)wait_teardown(last_commit, last_commit_parity);
  }
  if (*abort_flag && threadIdx.x == 0) atomicExch(p.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_short_tc(const ShortMaps &maps, const ShortGeom &g, const Problem &p,
                            void *out, int num_sms, cudaStream_t stream) {
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // setmaxnreg.inc only succeeds if the launch reserved the registers it hands
  // out; refuse to launch a build whose register count would not cover them.
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, attn_short_tc_kernel);
  if (e != cudaSuccess) return e;
  if (static_cast<long long>(fa.numRegs) * kThreads <
      2LL * 128 * kRegsSoftmax + 128LL * kRegsControl)
    return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(attn_short_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const int grid = g.units < num_sms ? g.units : num_sms;
  if (grid <= 0) return cudaSuccess;
  // programmatic dependent launch: this grid's set-up may overlap the end of
  // the previous kernel in the stream (the kernel waits before any global
  // memory access), and the next launch may do the same with this one
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_short_tc_kernel, maps, g, p, out);
}

}  // namespace mha
