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
// Warp roles (640 threads):
//   warps 0-15      four softmax warpgroups; unit n goes to warpgroup n % 4,
//                   thread t of a warpgroup owns tile row t
//   warp  16        TMA producer of Q and K (a 4-stage Q|K ring)
//   warp  17        TMA producer of V (a 4-stage V ring)
//   warp  18        TMEM owner and MMA issuer
//   warp  19        idle
// Per unit (the four steps of scaled dot-product attention):
//   S = Q K^T              tcgen05.mma -> the warpgroup's 128 TMEM columns
//   mask, scale, softmax   tcgen05.ld of the 32-column chunks the warp's rows
//                          can use -> registers; exp2 against the row max
//   P (bf16) -> TMEM       over the S columns already read
//   O = P V                tcgen05.mma (A = P from TMEM) -> the upper 64 of the
//                          warpgroup's columns
//   O / rowsum -> bf16     tcgen05.ld, 32 columns at a time; each warp stages
//                          its 32 half-rows in a swizzled 2 KiB buffer and
//                          writes them back, eight 64-byte pieces per store
// A Q|K stage is free once S is computed, a V stage once P V is: Q and K run
// ahead of the softmax independently of V.  The MMA warp issues whichever of
// the next S (its warpgroup free, Q and K landed) and the next P V (P
// posted, V landed) is ready.
// Padded sequences load only their first ceil(len/8)*8 rows, as one TMA box
// of that height per tensor and pair.  Before the dependency wait a CTA warms
// L2 with the whole tiles of its first two units: that traffic overlaps the
// previous grid's tail, when HBM would otherwise idle.
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
constexpr int kWGs = 4;                         // softmax warpgroups
constexpr int kStages = 4;                      // Q|K stages and V stages
constexpr int kTileRows = 128;
constexpr int kTileBytes = kTileRows * kD * 2;  // 16 KiB per operand tile
constexpr int kThreads = (kWGs + 1) * 128;      // 640
constexpr int kWgThreads = 128;
constexpr int kWarpProdQK = 4 * kWGs, kWarpProdV = kWarpProdQK + 1, kWarpMma = kWarpProdQK + 2;
// 640 threads at 96 registers each fill the register file; every role fits in
// 96 without spills, so no register split is needed.
constexpr uint32_t kTmemCols = 512;  // warpgroup w: [128 w, 128 w + 128)

struct __align__(8) Barriers {
  uint64_t qk_full[kStages], qk_empty[kStages];
  uint64_t v_full[kStages], v_empty[kStages];
  uint64_t s_full[kWGs];   // S of the warpgroup's unit is in TMEM
  uint64_t p_full[kWGs];   // the warpgroup read its S and wrote P
  uint64_t pv_done[kWGs];  // P V done: O ready
  uint64_t o_free[kWGs];   // the warpgroup read O: its columns are free
  uint64_t drain;          // teardown: every tcgen05 op of the CTA has finished
  uint32_t tmem_base;
  int abort_flag;
};

constexpr int kStagingBytes = 32 * 64;  // 32 output half-rows of one warp
constexpr size_t kSmemBytes = 1024 /* alignment slack */ + kStages * 2 * kTileBytes +
                              kStages * kTileBytes + 4 * kWGs * kStagingBytes + sizeof(Barriers);

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

// byte offset of 16-byte piece c (0..3) of 64-byte row `row` in a warp's
// staging buffer, swizzled so that eight consecutive lanes (one shared
// memory wavefront) never share a bank group, writing or reading
__device__ __forceinline__ uint32_t stage64_offset(uint32_t row, uint32_t c) {
  return row * 64u + ((c ^ ((row >> 1) & 3u)) << 4);
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
  uint8_t *qk_base = smem;                              // stage s: Q | K, 32 KiB
  uint8_t *v_base = qk_base + kStages * 2 * kTileBytes;  // stage s: V, 16 KiB
  uint8_t *staging = v_base + kStages * kTileBytes;     // 16 softmax warps x 2 KiB
  Barriers *bars = reinterpret_cast<Barriers *>(staging + 4 * kWGs * kStagingBytes);
  volatile int *abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int group = p.H / p.Hkv;  // query heads per key/value head
  // Causal 128-row tiles: row 96 + t needs four 32-key chunks of softmax,
  // row t one, and TMEM lanes 32 q .. 32 q + 31 belong to the warps on SM
  // sub-partition q.  Warpgroup w holds query-row block (j + w) % 4 in tile
  // rows 32 j .. 32 j + 31, so each sub-partition gets every kind of block.
  const bool rot = (p.mask & kMaskCausal) && g.Rq == 128 && !g.rows_q;
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const int n_local = c < g.units ? (g.units - 1 - c) / G + 1 : 0;

  // ---- setup -------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->qk_full[s], 1);
      mbar_init(&bars->qk_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int w = 0; w < kWGs; ++w) {
      mbar_init(&bars->s_full[w], 1);
      mbar_init(&bars->p_full[w], kWgThreads);
      mbar_init(&bars->pv_done[w], 1);
      mbar_init(&bars->o_free[w], kWgThreads);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpProdQK && lane == 0) {
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
  if (warp == kWarpMma) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // V rows that a padded unit does not load keep earlier contents; start
  // from zeros so they are always finite (their weights are exactly zero, and
  // 0 * NaN would not be).  Unloaded K and Q rows are masked by selection.
  if (g.rows_k) {
    for (int i = threadIdx.x; i < kStages * kTileBytes / 16; i += kThreads)
      reinterpret_cast<uint4 *>(v_base)[i] = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // Launched as a programmatic dependent, the kernel overlaps the previous
  // launch's tail up to griddep_wait: each role does its own set-up first and
  // waits just before its first global-memory access, so no warp's set-up
  // delays another's first copy once the dependency resolves.
  griddep_launch_dependents();

  int issued = 0;                   // producers: units whose loads were issued
  bool mma_issued = false;          // MMA issuer: a product was issued
  if (warp >= 4 * kWGs) {
   if (warp == kWarpProdQK || warp == kWarpProdV) {
    // ---- TMA producers (lane pp handles pair pp of the unit) ---------------
    const bool is_qk = warp == kWarpProdQK;
    const int pp = lane;
    const bool need_len = is_qk ? (g.rows_q || g.rows_k) : g.rows_k != 0;
    // lane l holds the length of unit n0 + l (all pairs of a unit share a
    // batch element); read 32 units at a time, well ahead of use
    auto load_lens = [&](int n0) -> int {
      const int nl = n0 + lane;
      if (!need_len || nl >= n_local) return 0;
      return clamp_len(p, (static_cast<int>(blockIdx.x) + nl * static_cast<int>(gridDim.x)) /
                              g.units_per_b);
    };
    UnitWalk cur(blockIdx.x, gridDim.x, g.units_per_b);
    griddep_wait();
    int lens = load_lens(0);
    for (int n = 0; n < n_local; ++n, cur.next()) {
      const int s = n % kStages;
      const int b = cur.b, h0 = cur.hu * g.P;
      // key/value head of pair pp (a pair past the last head, whose rows are
      // never stored, reads the last head so every box is in bounds)
      const int hq = min(h0 + pp, p.H - 1);
      const int hkv = group == 1 ? hq : hq / group;
      const bool rows_q = g.rows_q != 0, rows_k = g.rows_k != 0;
      const bool has_pair = pp < g.P && h0 + pp < p.H;
      if (n > 0 && (n & 31) == 0) lens = load_lens(n);
      const int len = __shfl_sync(0xffffffffu, lens, n & 31);
      // with unshared key/value heads the P pairs' first ceil8(len) key rows
      // come in as one box, packed back to back (see the softmax)
      const bool packed = rows_k && group == 1;
      uint32_t bytes = 0;
      if (is_qk && has_pair && rows_q) bytes += box_bytes(min(len, p.Lq));
      if (has_pair && rows_k && !packed) bytes += box_bytes(len);
      bytes = __reduce_add_sync(0xffffffffu, bytes);
      if (packed) bytes += g.P * box_bytes(len);
      if (is_qk && !rows_q) bytes += g.P * g.Rq * 128;
      if (!rows_k) bytes += g.P * g.Rk * 128;
      uint64_t *full = is_qk ? &bars->qk_full[s] : &bars->v_full[s];
      uint64_t *empty = is_qk ? &bars->qk_empty[s] : &bars->v_empty[s];
      if (!mbar_wait_warp(empty, ((n / kStages) & 1) ^ 1, abort_flag, p.wait_ns)) break;
      uint8_t *dq = qk_base + s * 2 * kTileBytes;  // Q tile (Q|K stage)
      uint8_t *dk = is_qk ? dq + kTileBytes : v_base + s * kTileBytes;  // K or V tile
      const CUtensorMap *kv_full = is_qk ? &maps.k_full : &maps.v_full;
      const CUtensorMap *kv_one = is_qk ? &maps.k_one : &maps.v_one;
      const CUtensorMap *kv_rows = is_qk ? maps.k_rows : maps.v_rows;
      if (lane == 0) mbar_arrive_expect_tx(full, bytes);
      __syncwarp();
      if (is_qk) {
        const int w = n % kWGs;
        if (rot && w != 0) {
          // rotated 32-row blocks (see above)
          if (lane < 4)
            tma_load_4d(dq + lane * 32 * 128, &maps.q_blk32, full, 0, ((lane + w) & 3) * 32, h0,
                        b);
        } else if (lane == 0 && !rows_q) {
          tma_load_4d(dq, &maps.q_full, full, 0, 0, h0, b);
        }
        if (has_pair && rows_q)
          load_rows(dq + pp * g.Rq * 128, maps.q_rows, full, min(len, p.Lq), h0 + pp, b);
      }
      // whole tiles: one box of P heads, or with shared key/value heads one
      // box per pair (heads past H read as zeros and are never stored)
      if (!rows_k && group == 1 && lane == 0) tma_load_4d(dk, kv_full, full, 0, 0, h0, b);
      if (!rows_k && group != 1 && pp < g.P)
        tma_load_4d(dk + pp * g.Rk * 128, kv_one, full, 0, 0, hkv, b);
      if (packed && lane == 0) load_rows(dk, kv_rows, full, len, h0, b);
      if (!packed && has_pair && rows_k)
        load_rows(dk + pp * g.Rk * 128, kv_rows, full, len, hkv, b);
      __syncwarp();
      issued = n + 1;
    }
   } else if (warp == kWarpMma) {
    // ---- MMA issuer (lane 0) ----------------------------------------------
    const uint32_t n_keys = static_cast<uint32_t>(g.P * g.Rk);  // multiple of 16, <= 128
    const uint32_t idesc_s = idesc_bf16_f32(128, n_keys, 0);
    const uint32_t idesc_o = idesc_bf16_f32(128, kD, 1);
    // S for unit ns needs its Q|K stage and its warpgroup's columns (free
    // once O of unit ns - 4 was read); P V for unit np needs P and the V
    // stage.  Issue whichever is ready; each stream stays in unit order.
    // Lane 0 alone polls the barriers and issues (tcgen05.mma and commit are
    // single-thread instructions); the other lanes wait at the end.  A wait
    // gives up after wait_ns without progress.
    if (lane == 0) {
      int ns = 0, np = 0;
      uint64_t t_idle = 0;  // start of the current stretch without progress
      uint32_t idle = 0;
      // test hook: a wait on a barrier that nothing signals before the teardown
      const bool run = !(p.stall & kStallShortMma) ||
                       mbar_wait(&bars->drain, 0, abort_flag, p.wait_ns);
      while (run && np < n_local) {
        bool did = false;
        if (ns < n_local) {
          const int s = ns % kStages, w = ns % kWGs;
          if (mbar_probe(&bars->qk_full[s], (ns / kStages) & 1) &&
              (ns < kWGs || mbar_probe(&bars->o_free[w], ((ns - kWGs) / kWGs) & 1))) {
            tc_fence_after();
            const uint32_t sq = smem_addr(qk_base + s * 2 * kTileBytes);
            const uint32_t sk = sq + kTileBytes;
  #pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              tc_mma_ss(tmem + w * 128, smem_desc_sw128(sq + kk * 32, 16, 1024),
                        smem_desc_sw128(sk + kk * 32, 16, 1024), idesc_s, kk > 0);
            tc_commit(&bars->s_full[w]);
            tc_commit(&bars->qk_empty[s]);
            mma_issued = true;
            ++ns;
            did = true;
          }
        }
        if (np < ns) {
          const int s = np % kStages, w = np % kWGs;
          if (mbar_probe(&bars->p_full[w], (np / kWGs) & 1) &&
              mbar_probe(&bars->v_full[s], (np / kStages) & 1)) {
            tc_fence_after();
            const uint32_t sv = smem_addr(v_base + s * kTileBytes);
            for (uint32_t kk = 0; kk < n_keys / 16; ++kk)
              // A = P (TMEM, 16 keys = 8 columns per step); B = V (MN-major)
              tc_mma_ts(tmem + w * 128 + 64, tmem + w * 128 + kk * 8,
                        smem_desc_sw128(sv + kk * 16 * 128, 1024, 1024), idesc_o, kk > 0);
            tc_commit(&bars->pv_done[w]);
            tc_commit(&bars->v_empty[s]);
            mma_issued = true;
            ++np;
            did = true;
          }
        }
        if (did) {
          t_idle = 0;
        } else if ((++idle & 63u) == 0) {
          const uint64_t now = global_timer_ns();
          if (t_idle == 0) t_idle = now;
          if (*abort_flag) break;
          if (now - t_idle > p.wait_ns) {
            *abort_flag = 1;
            break;
          }
        }
      }
    }
    __syncwarp();
   }
  } else {
    // ---- softmax + epilogue: warpgroup w takes units n = w, w + 4, ... -----
    const int w = warp >> 2;
    const int r = threadIdx.x & 127;  // tile row = TMEM lane
    const bool my_rot = rot && w != 0;  // query row of tile row r
    const int pr = r / g.Rq;
    const int i = my_rot ? ((((r >> 5) + w) & 3) << 5) | (r & 31) : r % g.Rq;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_tmem = tmem + lane_base + w * 128;  // S; P over its first 64
    const uint32_t o_tmem = s_tmem + 64;                 // O
    // a negative scale is applied as |scale| to sign-flipped scores.  Scores
    // are scaled after masking, so a zero scale would turn a masked -inf into
    // NaN; it is applied as the smallest normal float instead: every finite
    // score then flushes to 0 (exactly the zero-scale scores) and -inf stays
    const uint32_t sgn = p.scale_log2 < 0.f ? 0x80000000u : 0u;
    const float sl = p.scale_log2 != 0.f ? fabsf(p.scale_log2) : 1.17549435e-38f;
    const int rq_shift = __ffs(g.Rq) - 1;
    // byte strides of a query row and a head (below 2^31: this path takes
    // Lq <= 128 and H <= 2^24)
    const int row_stride = p.layout == kLayoutBHSD ? 128 : 128 * p.H;
    const int head_stride = p.layout == kLayoutBHSD ? 128 * p.Lq : 128;
    const long long batch_stride = 128LL * p.Lq * p.H;
    const uint32_t so = smem_addr(staging + warp * kStagingBytes);

    auto row_valid = [&](const UnitWalk &at) -> bool {
      return pr < g.P && at.hu * g.P + pr < p.H && i < p.Lq;
    };
    UnitWalk cur(blockIdx.x + w * gridDim.x, kWGs * gridDim.x, g.units_per_b);
    griddep_wait();
    int len_cur = (w < n_local && row_valid(cur)) ? clamp_len(p, cur.b) : 0;
    for (int n = w; n < n_local; n += kWGs) {
      const int k = n / kWGs;  // this warpgroup's k-th unit
      const bool valid = row_valid(cur);
      const int len = len_cur;
      int jmax = p.Lk;
      if (p.mask & kMaskKeyPadding) jmax = min(jmax, len);
      if (p.mask & kMaskCausal) jmax = min(jmax, i + 1);
      // cached decoding: query i sits at position len - Lq + i
      if (p.mask & kMaskCausalTail) jmax = max(min(jmax, len - p.Lq + i + 1), 0);
      const bool qpad = (p.mask & kMaskQueryPadding) && i >= len;
      if (!valid || qpad) jmax = 0;
      // key columns of this row's pair: packed units hold pair pr's keys at
      // [pr * ceil8(len), ...); whole-tile units (a CTA's first) at pr * Rk
      const bool packed = g.rows_k && group == 1;
      const int col_lo = pr * (packed ? ((len + 7) & ~7) : g.Rk);
      // 32-column chunks any row of this warp can use
      const unsigned lo = __reduce_min_sync(0xffffffffu, jmax > 0 ? col_lo : 1 << 20);
      const unsigned hi = __reduce_max_sync(0xffffffffu, jmax > 0 ? col_lo + jmax : 0);
      const int ch_lo = hi > 0 ? static_cast<int>(lo / 32) : 4;
      const int ch_hi = hi > 0 ? static_cast<int>((hi + 31) / 32) : 0;

      if (!mbar_wait_warp(&bars->s_full[w], k & 1, abort_flag, p.wait_ns)) break;
      tc_fence_after();
      // keep only this row's keys [col_lo, col_lo + jmax).  One pass over
      // the chunks: exponents are taken against the first chunk's max m;
      // a later chunk may exceed m by up to 2^8 (P stays far from bf16
      // overflow, and numerator and denominator share m, so the quotient
      // is unchanged).  A row whose max grows further rescales the P it
      // already wrote (rare: the scores would have to climb steeply along
      // the keys).  P of chunk ch goes to columns [16 ch, 16 ch + 16), which
      // hold scores already read.
      const int lo_c = col_lo, hi_c = col_lo + jmax;
      float ms = -INFINITY;  // reference max, scaled (log2 units)
      float rowsum = 0.f;
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
            for (int c = ch_lo; c < ch; ++c) rescale_p(s_tmem + c * 16, f);
            if (climb) ms = cm;
          }
          rowsum += chunk_exp_pack(v, sl, ms == -INFINITY ? 0.f : ms, pk);
        } else {
#pragma unroll
          for (int t = 0; t < 16; ++t) pk[t] = 0u;
        }
        tmem_st16(s_tmem + ch * 16, pk);
      }
      const bool zero_row = ms == -INFINITY;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full[w]);

      // ---- epilogue: O / rowsum -> bf16 -> global, 32 columns at a time ----
      if (!mbar_wait_warp(&bars->pv_done[w], k & 1, abort_flag, p.wait_ns)) break;
      tc_fence_after();
      const float inv = zero_row ? 0.f : 1.f / rowsum;
      const int b = cur.b, h0 = cur.hu * g.P;
      if (p.lse != nullptr && valid)
        p.lse[(static_cast<size_t>(b) * p.H + h0 + pr) * p.Lq + i] =
            zero_row ? INFINITY : ms + __log2f(rowsum);
      uint8_t *obase = static_cast<uint8_t *>(out) + b * batch_stride;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t o[32];
        tmem_ld32(o_tmem + 32 * half, o);
        tmem_wait_ld();
        if (half == 1) {
          tc_fence_before();
          mbar_arrive(&bars->o_free[w]);
        }
        // this lane's row, 64 bytes, into the warp's staging rows
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t wv[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int c = c4 * 8 + 2 * t;
            wv[t] = zero_row ? 0u
                             : pack_bf16x2(__uint_as_float(o[c]) * inv,
                                           __uint_as_float(o[c + 1]) * inv);
          }
          st_shared_v4(so + stage64_offset(lane, c4), wv[0], wv[1], wv[2], wv[3]);
        }
        __syncwarp();
        // eight rows per store instruction, 64 contiguous bytes of each
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int rr = 8 * t + (lane >> 2);   // warp row
          const int row = (warp & 3) * 32 + rr;  // tile row
          const int pr_o = row >> rq_shift;
          const int i_o = my_rot ? ((((row >> 5) + w) & 3) << 5) | (row & 31) : row & (g.Rq - 1);
          const uint4 val = ld_shared_v4(so + stage64_offset(rr, lane & 3));
          if (pr_o < g.P && h0 + pr_o < p.H && i_o < p.Lq)
            st_global_v4(obase + static_cast<long long>(h0 + pr_o) * head_stride +
                             static_cast<long long>(i_o) * row_stride + half * 64 + (lane & 3) * 16,
                         val);
        }
        __syncwarp();
      }
      // the next unit's length, loaded while its scores are computed
      cur.next();
      len_cur = (n + kWGs < n_local && row_valid(cur)) ? clamp_len(p, cur.b) : 0;
    }
  }

  // ---- teardown ------------------------------------------------------------
  if (*abort_flag && (warp == kWarpProdQK || warp == kWarpProdV) && lane == 0) {
    // let copies already in flight land before the CTA's shared memory goes away
    uint64_t *fulls = warp == kWarpProdQK ? bars->qk_full : bars->v_full;
    for (int n = issued - kStages; n < issued; ++n)
      if (n >= 0) (void)wait_teardown(&fulls[n % kStages], (n / kStages) & 1);
  }
  if (*abort_flag && warp == kWarpMma && lane == 0 && mma_issued) {
    // tcgen05 ops of one thread complete in order: one more commit covers
    // every product issued before it
    tc_commit(&bars->drain);
    (void)wait_teardown(&bars->drain, 0);
  }
  if (*abort_flag && threadIdx.x == 0) atomicExch(p.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_short_tc(const ShortMaps &maps, const ShortGeom &g, const Problem &p,
                            void *out, int num_sms, cudaStream_t stream) {
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(attn_short_tc_kernel),
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
