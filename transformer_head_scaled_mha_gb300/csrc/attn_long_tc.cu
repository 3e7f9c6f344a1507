// Long-sequence attention on the tcgen05 tensor cores (bf16, d in {64, 128}).
//
// One CTA computes 256 query rows of one (batch, head) as two 128-row tiles,
// one per softmax warpgroup, streaming the keys/values in 128-row tiles:
//
//   S_w = Q_w K_j^T          tcgen05.mma, both operands from 128B-swizzled
//                            smem, fp32 accumulator in TMEM (one 128-column
//                            region per warpgroup)
//   online softmax           tcgen05.ld of S into registers (thread = row),
//                            scale folded with log2(e), causal / padding mask
//                            on the tiles that straddle a boundary, running max
//                            and running sum; exp2 on the MUFU unit
//   P_w (bf16) -> TMEM       tcgen05.st over the first 64 columns of S_w
//   O_w += P_w V_j           tcgen05.mma with A = P_w read from TMEM, B = V_j
//                            from smem, fp32 accumulator in TMEM
//   epilogue                 O / rowsum -> bf16 -> swizzled smem -> TMA store
//
// The score matrix never leaves the SM.  While one warpgroup turns its S into
// P, the tensor core runs the other warpgroup's products (ping-pong).  Per
// warpgroup the MMA warp issues P_w(j-1) V_{j-1} before S_w(j) (the tensor
// pipe runs one thread's MMAs in order, so S_w(j) overwrites P_w(j-1) only
// after it was read), and the commit that announces S_w(j) also covers
// P_w(j-1) V_{j-1}, so a warpgroup holding S_w(j) may rescale O_w at once.
// K and V stream through a ring of smem slots two iterations ahead of use.
// The running max is moved (and O rescaled in TMEM) only when it grows by more
// than 2^8; numerator and denominator share the stale max, so the quotient is
// unchanged.  Under a causal mask the tiles above the diagonal are never
// loaded nor multiplied, which halves the work; CTAs are issued in bands of
// query blocks, heaviest band first, a head's blocks of a band together.
//
// Warp roles (384 threads): warps 0-3 softmax WG0, 4-7 softmax WG1, warp 8 TMA
// producer, warp 9 TMEM owner + MMA issuer, warps 10-11 idle (they complete the
// third warpgroup so its register budget can be handed to the softmax).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int kBM = 128;  // query rows per warpgroup tile
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kThreads = 384;  // 3 warpgroups
constexpr int kWgThreads = 128;
// Register split: launched at 168 per thread (384 x 168 = 64512); the
// producer/MMA warpgroup drops to 56 and the two softmax warpgroups rise to
// 224: 2 x 128 x 224 + 128 x 56 = 64512.
constexpr uint32_t kRegsSoftmax = 224;
constexpr uint32_t kRegsControl = 56;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsControl <= kThreads * 168, "register split");
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: O may grow to 2^8 before a rescale
constexpr int kMaxSlots = 8;
constexpr int kBand = 8;  // query blocks per band of the CTA order

template <int D>
struct Cfg {
  static constexpr int kBlkBytes = 128 * 128;              // one [128 rows x 64] swizzle block
  static constexpr int kTileBytes = (D / 64) * kBlkBytes;  // a [128 x D] operand tile
  static constexpr int kSlots = (D == 128) ? 5 : 8;        // K/V ring (K0 V0 K1 V1 ...)
  static constexpr size_t kSmem = 1024 + 2 * kTileBytes + kSlots * kTileBytes + 256;
};

struct __align__(8) Barriers {
  uint64_t q_full;
  uint64_t kv_full[kMaxSlots];
  uint64_t kv_empty[kMaxSlots];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t drain;  // teardown: every tcgen05 op of the CTA has finished
  uint32_t tmem_base;
  int abort_flag;
};

// share of the exponentials of an unmasked chunk taken on the FMA pipes
// (exp2_poly2) instead of the MUFU unit: pairs k of the chunk with
// k % kPolyEvery == kPolyEvery - 1 (0: none)
constexpr int kPolyEvery = 0;

// Row maximum of one 32-column chunk (raw fp32 bits); a tree of 3-input
// maxima, depth 4.
__device__ __forceinline__ float chunk_max32(const uint32_t (&v)[32]) {
  float t[11];
#pragma unroll
  for (int k = 0; k < 10; ++k)
    t[k] = fmax3(__uint_as_float(v[3 * k]), __uint_as_float(v[3 * k + 1]),
                 __uint_as_float(v[3 * k + 2]));
  t[10] = fmaxf(__uint_as_float(v[30]), __uint_as_float(v[31]));
  return fmax3(fmax3(t[0], t[1], t[2]), fmax3(t[3], t[4], t[5]),
               fmax3(fmax3(t[6], t[7], t[8]), t[9], t[10]));
}

// p_c = exp2(s_c * sl - m) for one 32-column chunk, packed into 16 bf16x2
// columns; returns the chunk's sum of p (fp32)
__device__ __forceinline__ float chunk_exp_pack32(const uint32_t (&v)[32], float sl, float m,
                                                  uint32_t (&pk)[16]) {
  const uint64_t sc = f2_pack(sl, sl);
  const uint64_t nm = f2_pack(-m, -m);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float a, b;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sc, nm), a, b);
    if (kPolyEvery > 0 && (e >> 1) % (kPolyEvery > 0 ? kPolyEvery : 1) == kPolyEvery - 1) {
      exp2_poly2(a, b);
    } else {
      a = ex2_approx(a);
      b = ex2_approx(b);
    }
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

// Multiplies the 32 bf16 P values of one chunk (16 TMEM columns) by f, after
// the stores in flight have landed.
__device__ __noinline__ void rescale_p16(uint32_t taddr, float f) {
  uint32_t r[16];
  tmem_wait_st();
  tmem_ld16(taddr, r);
  tmem_wait_ld();
#pragma unroll
  for (int t = 0; t < 16; ++t)
    r[t] = pack_bf16x2(__uint_as_float(r[t] << 16) * f, __uint_as_float(r[t] & 0xffff0000u) * f);
  tmem_st16(taddr, r);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_long_tc_kernel(const __grid_constant__ LongMaps maps, const Problem p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *q_smem = smem;                         // 2 tiles; reused as output staging
  uint8_t *kv_smem = q_smem + 2 * C::kTileBytes;  // kSlots tiles
  Barriers *bars = reinterpret_cast<Barriers *>(kv_smem + C::kSlots * C::kTileBytes);
  volatile int *abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BH = p.B * p.H;
  const int nqb = (p.Lq + 2 * kBM - 1) / (2 * kBM);
  // CTA order: bands of kBand query blocks, heaviest band first; inside a
  // band, all its query blocks of one head side by side (heaviest first), so
  // the CTAs running at one time that read a head's keys and values read the
  // same tiles at about the same time and mostly find them in L2
  int qb, bh;
  {
    const int x = static_cast<int>(blockIdx.x);
    const int full = nqb / kBand;  // full bands; a partial one (the lightest) ends the order
    const int t = min(x / (BH * kBand), full);
    const int hi = nqb - t * kBand;  // the band's query blocks are [hi - size, hi)
    const int size = min(kBand, hi);
    const int local = x - t * BH * kBand;
    bh = local / size;
    qb = hi - 1 - local % size;
  }
  const int b = bh / p.H, h = bh % p.H;
  const int hkv = h / (p.H / p.Hkv);  // key/value head this query head reads
  const int q0 = qb * 2 * kBM;

  int len = p.Lk;
  if (p.mask & (kMaskKeyPadding | kMaskQueryPadding)) {
    const int l = p.key_lengths[b];
    len = l < 0 ? 0 : (l > p.Lk ? p.Lk : l);
  }
  // warpgroup w owns rows [q0 + 128 w, +128) and needs key tiles [0, n_tiles[w])
  int n_tiles[2];
  bool wg_rows[2];
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    const int r0 = q0 + w * kBM;
    wg_rows[w] = r0 < p.Lq;
    int kv_end = p.Lk;
    if (p.mask & kMaskKeyPadding) kv_end = min(kv_end, len);
    if (p.mask & kMaskCausal) kv_end = min(kv_end, min(r0 + kBM, p.Lq));
    // the tile's last query sits at position len - Lq + its row
    if (p.mask & kMaskCausalTail) kv_end = min(kv_end, len - p.Lq + min(r0 + kBM, p.Lq));
    n_tiles[w] = wg_rows[w] && kv_end > 0 ? (kv_end + kBN - 1) / kBN : 0;
  }
  const int n_kv = max(n_tiles[0], n_tiles[1]);

  // ---- setup -------------------------------------------------------------
  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&bars->s_full[w], 1);
      mbar_init(&bars->p_full[w], kWgThreads);
      mbar_init(&bars->pv_done[w], 1);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  // TMEM columns: S_w / P_w at [128 w, 128 w + 128), O_w at [256 + 128 w, +D)

  int issued = 0;           // producer: K/V loads issued
  bool mma_issued = false;  // MMA lane: a product was issued

  if (warp >= 8) {
   regs_dec<kRegsControl>();
   if (warp == 8) {
    // ---- TMA producer: Q tiles, then K_0 V_0 K_1 V_1 ... through the ring --
    if (lane == 0 && n_kv > 0) {
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      uint32_t qbytes = 0;
      for (int w = 0; w < 2; ++w)
        if (n_tiles[w] > 0) qbytes += C::kTileBytes;
      mbar_arrive_expect_tx(&bars->q_full, qbytes);
      for (int w = 0; w < 2; ++w)
        if (n_tiles[w] > 0)
          for (int blk = 0; blk < D / 64; ++blk)
            tma_load_4d(q_smem + w * C::kTileBytes + blk * C::kBlkBytes, &maps.q, &bars->q_full,
                        blk * 64, q0 + w * kBM, h, b);
      for (int idx = 0; idx < 2 * n_kv; ++idx) {
        const int slot = idx % C::kSlots, round = idx / C::kSlots;
        if (!mbar_wait(&bars->kv_empty[slot], (round & 1) ^ 1, abort_flag, p.wait_ns)) break;
        const int j = idx >> 1;
        const CUtensorMap *map = (idx & 1) ? &maps.v : &maps.k;
        mbar_arrive_expect_tx(&bars->kv_full[slot], C::kTileBytes);
        for (int blk = 0; blk < D / 64; ++blk)
          tma_load_4d(kv_smem + slot * C::kTileBytes + blk * C::kBlkBytes, map,
                      &bars->kv_full[slot], blk * 64, j * kBN, hkv, b);
        issued = idx + 1;
      }
    }
  } else if (warp == 9) {
    // ---- MMA issuer: lane 0 alone (tcgen05.mma and commit are single-thread
    // instructions); the other lanes wait at the end --------------------------
    // iteration j, per warpgroup w: O_w += P_w(j-1) V_{j-1}, then S_w(j) = Q_w K_j^T.
    // The K/V slots are released by the warpgroup whose S_w(j) comes last
    // (its commit covers every earlier product), which spares this thread
    // two commits per iteration.
    if (lane == 0) {
      const uint32_t idesc_s = idesc_bf16_f32(128, kBN, 0);
      const uint32_t idesc_o = idesc_bf16_f32(128, D, 1);
      constexpr uint32_t kVLbo = C::kBlkBytes, kVSbo = 1024;
      // descriptors: a constant high half, a low half stepped per piece
      const uint32_t hi_s = smem_desc_hi(1024), hi_v = smem_desc_hi(kVSbo);
      const uint32_t q_lo[2] = {smem_desc_lo(smem_addr(q_smem), 16),
                                smem_desc_lo(smem_addr(q_smem + C::kTileBytes), 16)};
      const uint32_t kv_lo = smem_desc_lo(smem_addr(kv_smem), 16);
      const uint32_t v_lo = smem_desc_lo(smem_addr(kv_smem), kVLbo);
      constexpr uint32_t kSlotLo = C::kTileBytes >> 4;  // low-half step between ring slots
      // ring position of K_j (index 2 j) and V_{j-1} (index 2 j - 1): slot
      // and round, stepped without divisions
      int ks = 0, kr = 0, vs = 0, vr = 0;
      bool ok = n_kv == 0 || mbar_wait(&bars->q_full, 0, abort_flag, p.wait_ns);
      for (int j = 0; ok && j <= n_kv; ++j) {
        // test hook: a wait on a barrier that nothing signals before the
        // teardown, with products and copies in flight
        if ((p.stall & kStallLongMma) && j == 2 &&
            !(ok = mbar_wait(&bars->drain, 0, abort_flag, p.wait_ns)))
          break;
        if (j < n_kv && !(ok = mbar_wait_spin(&bars->kv_full[ks], kr & 1, abort_flag, p.wait_ns)))
          break;
        if (j >= 1 && !(ok = mbar_wait_spin(&bars->kv_full[vs], vr & 1, abort_flag, p.wait_ns)))
          break;
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          const bool do_pv = j >= 1 && j - 1 < n_tiles[w];
          const bool do_s = j < n_tiles[w];
          if (do_pv &&
              !(ok = mbar_wait_spin(&bars->p_full[w], (j - 1) & 1, abort_flag, p.wait_ns)))
            break;
          tc_fence_after();
          if (do_pv) {
            const uint32_t lo = v_lo + vs * kSlotLo;
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              // B = V_{j-1}, MN-major: 16 key rows per step (8-row groups 1024 B
              // apart); its D/64 blocks of 64 value columns lie kBlkBytes apart.
              // A = P_w(j-1): 16 keys = 8 TMEM columns per step
              tc_mma_ts(tmem + 256 + w * 128, tmem + w * 128 + kk * 8,
                        desc_join(lo + ((kk * 16 * 128) >> 4), hi_v), idesc_o,
                        (j - 1 > 0) || kk > 0);
            // only the epilogue waits for P V on its own, after the last
            // one; every earlier P V is covered by the next S's commit
            if (j == n_tiles[w]) tc_commit(&bars->pv_done[w]);
            mma_issued = true;
          }
          if (do_s) {
            const uint32_t lo = kv_lo + ks * kSlotLo;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = ((kk >> 2) * C::kBlkBytes + (kk & 3) * 32) >> 4;
              tc_mma_ss(tmem + w * 128, desc_join(q_lo[w] + off, hi_s),
                        desc_join(lo + off, hi_s), idesc_s, kk > 0);
            }
            tc_commit(&bars->s_full[w]);
            mma_issued = true;
          }
        }
        // next iteration: K_{j+1} at index 2 j + 2, V_j at 2 j + 1
        vs = ks + 1;
        vr = kr;
        if (vs == C::kSlots) {
          vs = 0;
          ++vr;
        }
        ks += 2;
        if (ks >= C::kSlots) {
          ks -= C::kSlots;
          ++kr;
        }
      }
    }
    __syncwarp();
   }
  } else {
    regs_inc<kRegsSoftmax>();
    // ---- softmax warpgroups --------------------------------------------------
    const int w = warp >> 2;           // warpgroup
    const int r = threadIdx.x & 127;   // row within the tile (TMEM lane)
    const int i = q0 + w * kBM + r;    // query row
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_tmem = tmem + lane_base + w * 128;
    const uint32_t o_tmem = tmem + lane_base + 256 + w * 128;
    const int nt = n_tiles[w];
    int jmax = p.Lk;  // keys j < jmax are allowed for row i
    if (p.mask & kMaskKeyPadding) jmax = min(jmax, len);
    if (p.mask & kMaskCausal) jmax = min(jmax, i + 1);
    if (p.mask & kMaskCausalTail) jmax = max(min(jmax, len - p.Lq + i + 1), 0);
    const bool qpad = (p.mask & kMaskQueryPadding) && i >= len;

    float m_use = -INFINITY;  // max used for the exponentials (log2 units)
    float l_run = 0.f;
    bool ok = true;
    // the warpgroup with the most key tiles (WG1, unless its rows lie past
    // the end) releases the K/V slots: once it holds S_w(j), every product
    // issued before -- both warpgroups' reads of K_j and V_{j-1} -- is done
    const bool releaser = w == (wg_rows[1] ? 1 : 0);
    for (int j = 0; j < nt; ++j) {
      // S_w(j) is ready, and so is P_w(j-1) V_{j-1} (same commit)
      if (!(ok = mbar_wait_warp(&bars->s_full[w], j & 1, abort_flag, p.wait_ns))) break;
      tc_fence_after();
      if (releaser && r == 0) {
        mbar_arrive(&bars->kv_empty[(2 * j) % C::kSlots]);
        if (j >= 1) mbar_arrive(&bars->kv_empty[(2 * j - 1) % C::kSlots]);
      }
      // columns c < lim are allowed; a row may allow none of this tile's
      // columns (rows of one tile see different key counts under the
      // cached-decoding mask), so clamp to [0, kBN]
      const int lim = min(max(jmax - j * kBN, 0), kBN);
      const bool need_mask = __any_sync(0xffffffffu, lim < kBN);
      const bool pos = p.scale_log2 > 0.f;
      float alpha = 1.f;
      if (pos && !need_mask && __all_sync(0xffffffffu, m_use != -INFINITY)) {
        // Unmasked tile, every row of the warp has a running max: 32-column
        // chunks, exponents against the running max; all four chunks' TMEM
        // loads go out at once (one wait instead of one per chunk).  A chunk
        // whose max exceeds the running max by more than 2^8 moves it first
        // (and rescales the P of the chunks already stored).  P of chunk ch
        // goes to columns [16 ch, 16 ch + 16), whose scores are already read.
        uint32_t vall[4][32];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) tmem_ld32(s_tmem + ch * 32, vall[ch]);
        tmem_wait_ld();
        float tsum = 0.f;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t(&cur)[32] = vall[ch];
          const float cm = chunk_max32(cur) * p.scale_log2;
          const bool climb = cm > m_use + kRescaleThreshold;
          if (__any_sync(0xffffffffu, climb)) {
            const float f = climb ? ex2_approx(m_use - cm) : 1.f;
            if (climb) m_use = cm;
            alpha *= f;
            tsum *= f;
#pragma unroll 1
            for (int c = 0; c < ch; ++c) rescale_p16(s_tmem + c * 16, f);
          }
          uint32_t pk[16];
          tsum += chunk_exp_pack32(cur, p.scale_log2, m_use, pk);
          tmem_st16(s_tmem + ch * 16, pk);
        }
        l_run = l_run * alpha + tsum;
      } else {
        uint32_t sr[4][32];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) tmem_ld32(s_tmem + ch * 32, sr[ch]);
        tmem_wait_ld();
        // positive scale: max over the raw scores, then one FMA per score;
        // otherwise scale first (the max of scale * s is not scale * max s)
        const float mt = pos ? mask_max128(sr, need_mask, 0, lim) * p.scale_log2
                             : scale_mask_max128(sr, p.scale_log2, need_mask, 0, lim);
        const float m_new = fmaxf(m_use, mt);
        if (m_new > m_use + kRescaleThreshold) {
          if (m_use != -INFINITY) alpha = ex2_approx(m_use - m_new);
          m_use = m_new;
        }
        const bool live = m_use != -INFINITY;
        l_run = l_run * alpha + (pos ? exp2_fma_sum128(sr, p.scale_log2, m_use, live)
                                     : exp2_sum128(sr, m_use, live));
        // P_w(j) as bf16 pairs over the first 64 columns of S_w
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            const int c = h * 64 + 2 * t;
            pk[t] = pack_bf16x2(__uint_as_float(sr[c >> 5][c & 31]),
                                __uint_as_float(sr[c >> 5][(c + 1) & 31]));
          }
          tmem_st32(s_tmem + h * 32, pk);
        }
      }
      // the running max moved: rescale this row of O (rare, warp-wide)
      if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(o_tmem + ch * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(o_tmem + ch * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full[w]);
    }

    // ---- epilogue: O / l -> bf16 -> staging (this warpgroup's Q tile) -> TMA
    // (the decision to store is taken by the whole warpgroup at once: its
    // warps meet at a named barrier below, which a warp that gave up would
    // never reach)
    if (ok && nt > 0) ok = mbar_wait_warp(&bars->pv_done[w], 0, abort_flag, p.wait_ns);
    ok = named_barrier_and(1 + w, kWgThreads, ok);
    if (ok && wg_rows[w]) {
      const bool zero_row = qpad || l_run == 0.f || nt == 0;
      const float inv = zero_row ? 0.f : 1.f / l_run;
      if (p.lse != nullptr && i < p.Lq)
        p.lse[(static_cast<size_t>(b) * p.H + h) * p.Lq + i] =
            zero_row ? INFINITY : m_use + __log2f(l_run);
      if (nt > 0) tc_fence_after();
      {
        uint8_t *stage = q_smem + w * C::kTileBytes;
        const uint32_t so = smem_addr(stage);
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          if (nt > 0) {
            tmem_ld32(o_tmem + ch * 32, o);
            tmem_wait_ld();
          }
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t wv[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const float a0 = zero_row ? 0.f : __uint_as_float(o[q4 * 8 + 2 * t]) * inv;
              const float a1 = zero_row ? 0.f : __uint_as_float(o[q4 * 8 + 2 * t + 1]) * inv;
              wv[t] = pack_bf16x2(a0, a1);
            }
            const int c16 = ch * 4 + q4;  // 16-byte piece within the row
            st_shared_v4(so + (c16 >> 3) * C::kBlkBytes + sw128_offset(r, c16 & 7), wv[0],
                         wv[1], wv[2], wv[3]);
          }
        }
        fence_proxy_async_smem();
        named_barrier_sync(1 + w, kWgThreads);
        if (r == 0) {
          for (int blk = 0; blk < D / 64; ++blk)
            tma_store_4d(&maps.o, stage + blk * C::kBlkBytes, blk * 64, q0 + w * kBM, h, b);
          tma_store_commit();
          tma_store_wait0();
        }
      }
    }
  }

  // ---- teardown --------------------------------------------------------------
  if (*abort_flag && warp == 8 && lane == 0) {
    for (int idx = issued - C::kSlots; idx < issued; ++idx)
      if (idx >= 0) (void)wait_teardown(&bars->kv_full[idx % C::kSlots], (idx / C::kSlots) & 1);
    if (n_kv > 0) (void)wait_teardown(&bars->q_full, 0);
  }
  if (*abort_flag && warp == 9 && lane == 0 && mma_issued) {
    // tcgen05 ops of one thread complete in order: one more commit covers
    // every product issued before it
    tc_commit(&bars->drain);
    (void)wait_teardown(&bars->drain, 0);
  }
  if (*abort_flag && threadIdx.x == 0) atomicExch(p.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, kTmemCols);
}

template <int D>
cudaError_t launch_long_impl(const LongMaps &maps, const Problem &p, cudaStream_t stream) {
  static_assert(Cfg<D>::kSmem <= 232448, "shared memory budget");
  static_assert(Cfg<D>::kSlots <= kMaxSlots, "ring size");
  // setmaxnreg.inc only succeeds if the launch reserved the registers it hands
  // out; refuse to launch a build whose register count would not cover them.
  // (checked once per process: the register count is a property of the build)
  static std::atomic<int> regs_ok{0};  // 0 unknown, 1 enough, 2 too few
  if (regs_ok.load(std::memory_order_acquire) == 0) {
    cudaFuncAttributes fa;
    const cudaError_t e = cudaFuncGetAttributes(&fa, attn_long_tc_kernel<D>);
    if (e != cudaSuccess) return e;
    regs_ok.store(static_cast<long long>(fa.numRegs) * kThreads >=
                          2LL * 128 * kRegsSoftmax + 128LL * kRegsControl
                      ? 1
                      : 2,
                  std::memory_order_release);
  }
  if (regs_ok.load(std::memory_order_acquire) != 1) return cudaErrorInvalidConfiguration;
  cudaError_t e = set_smem_once(reinterpret_cast<const void *>(attn_long_tc_kernel<D>),
                                static_cast<int>(Cfg<D>::kSmem));
  if (e != cudaSuccess) return e;
  const int nqb = (p.Lq + 2 * kBM - 1) / (2 * kBM);
  const long long grid = static_cast<long long>(p.B) * p.H * nqb;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  attn_long_tc_kernel<D><<<static_cast<unsigned>(grid), kThreads, Cfg<D>::kSmem, stream>>>(maps, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_long_tc(const LongMaps &maps, const Problem &p, int num_sms,
                           cudaStream_t stream) {
  (void)num_sms;
  if (p.dk == 128) return launch_long_impl<128>(maps, p, stream);
  return launch_long_impl<64>(maps, p, stream);
}

}  // namespace mha
