// Shared definitions between the host dispatcher and the kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mha {

constexpr int kMaskCausal = 1;
constexpr int kMaskKeyPadding = 2;
constexpr int kMaskQueryPadding = 4;
constexpr int kMaskCausalTail = 8;  // queries are the last Lq of len keys (cached decoding)

constexpr int kStatusOk = 0;
constexpr int kStatusTimeout = 4;

// A bounded wait gives up after this much wall time.  Every wait in these
// kernels normally completes within microseconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// log2(e): softmax is evaluated as exp2(x * scale * log2(e) - m)
constexpr float kLog2e = 1.4426950408889634f;

constexpr int kLayoutBHSD = 0;  // [B, heads, L, d]
constexpr int kLayoutBSHD = 1;  // [B, L, heads, d]

// Problem description handed to every kernel by value.
struct Problem {
  int B, H, Hkv, Lq, Lk, dk, dv;  // query head h reads key/value head h / (H / Hkv)
  int layout;                      // kLayoutBHSD or kLayoutBSHD (all four tensors)
  int mask;
  const int32_t *key_lengths;  // device [B] or nullptr
  float scale_log2;            // scale * log2(e)
  int *status;                 // device status word (kStatusTimeout on a given-up wait)
  uint64_t wait_ns;            // a bounded wait gives up after this long
  int stall;                   // test hook: kStall* bits make a kernel wait on a barrier
                               // that nothing signals (0 in normal use)
  float *lse;                  // device [B, H, Lq] or nullptr: each row's log2 of the
                               // softmax denominator of the scaled scores (+inf for a
                               // row stored as zeros), for the backward pass
};

// Test hooks for the give-up path of the bounded waits (Problem::stall).
constexpr int kStallShortMma = 1;  // short kernel: the MMA issuer waits before its first product
constexpr int kStallLongMma = 2;   // long kernel: the MMA issuer waits before its third iteration

// Sets the dynamic shared-memory limit of a kernel once per device context
// (a driver call per launch costs host time on every call).
cudaError_t set_smem_once(const void *kernel, int bytes);

// ---- kernel launchers (defined next to each kernel) ----------------------
cudaError_t launch_f32_simt(const float *q, const float *k, const float *v, float *out,
                            const Problem &p, cudaStream_t stream);

// tensor maps for the bf16 tensor-core kernels: every map is 4-D
// (d, L, heads, B) over a bf16 tensor in either layout, 128-byte swizzle
constexpr int kRowBoxes = 16;  // row-box heights 8, 16, ..., 128
struct ShortMaps {
  CUtensorMap q_full;                  // box (64, Rq, P, 1): P consecutive query heads
  CUtensorMap k_full, v_full;          // box (64, Rk, P, 1) (key/value heads not shared)
  CUtensorMap k_one, v_one;            // box (64, Rk, 1, 1) (shared key/value heads)
  CUtensorMap q_rows[kRowBoxes];       // box (64, 8 (h + 1), 1, 1), for padded tensors
  CUtensorMap k_rows[kRowBoxes];       // box (64, 8 (h + 1), P, 1) (1 head if shared)
  CUtensorMap v_rows[kRowBoxes];
  CUtensorMap q_blk32;                 // box (64, 32, 1, 1): causal row-block order
};
struct ShortGeom {
  int Rq, Rk, P;       // rows per packed pair (powers of two) and pairs per unit
  int units_per_b;     // ceil(H / P): a unit never spans two batch elements
  int units;           // B * units_per_b
  int rows_q, rows_k;  // load Q / K,V only up to each pair's length (padding)
  const void *q, *k, *v;  // the tensors themselves (L2 prefetch by address)
};
cudaError_t launch_short_tc(const ShortMaps &maps, const ShortGeom &g, const Problem &p,
                            void *out, int num_sms, cudaStream_t stream);

struct LongMaps {
  CUtensorMap q, k, v;  // box (64, 128, 1, 1)
  CUtensorMap o;        // box (64, 128, 1, 1)
};
cudaError_t launch_long_tc(const LongMaps &maps, const Problem &p, int num_sms,
                           cudaStream_t stream);

// few query rows (R = (H / Hkv) * Lq <= 16) against many keys: Q box
// (64, Lq, H / Hkv, 1) -- a key/value head's whole group of query heads --,
// K and V boxes (64, 128, 1, 1)
struct DecodeMaps {
  CUtensorMap q, k, v;
};
cudaError_t launch_decode_tc(const DecodeMaps &maps, const Problem &p, void *out, int num_sms,
                             cudaStream_t stream);

// backward pass: tensors in the forward's layout and dtype; lse and dsum
// (D = dout . out) are fp32 per query row [B * H * Lq], lse in log2 units of
// the scaled scores (+inf for a row that attends to nothing)
struct BwdArgs {
  const void *q, *k, *v, *out, *dout;
  void *dq, *dk, *dv;
  float *lse, *dsum;
  float scale;  // dq and dk carry this factor
  // d = 64 with query and key lengths <= 128: (batch, head) pairs packed per
  // 128-row tile by the fused short kernel (its maps have box (64, 128 /
  // pack, pack, 1)); 1 otherwise
  int pack;
};
cudaError_t launch_bwd_simt(const BwdArgs &a, const Problem &p, bool bf16, cudaStream_t stream);
// D = dout . out per query row into a.dsum (bf16 tensors), when the row
// statistics lse come from the forward pass instead of a statistics pass
cudaError_t launch_bwd_dsum(const BwdArgs &a, const Problem &p, cudaStream_t stream);
// bf16, d in {64, 128}: maps q, k, v and (in the `o` slot) dout, box
// (64, 128, 1, 1), or (64, 128 / a.pack, a.pack, 1) for the fused short kernel
cudaError_t launch_bwd_tc(const LongMaps &maps, const Problem &p, const BwdArgs &a, int num_sms,
                          cudaStream_t stream, bool have_lse = false);

cudaError_t launch_zero_fill(void *out, size_t bytes, cudaStream_t stream);
// dst[0, n) = value
cudaError_t launch_fill_f32(float *dst, size_t n, float value, cudaStream_t stream);

// y_g = x_g W_g + b_g (bf16) for up to kMaxLinear products with the same K in
// one launch, 128-byte swizzle.  Slab tiling (K and every N multiples of 64):
// x viewed as (64, M, K/64) box (64, 128, 2), W as (64, K, N/64) box
// (64, 128, 2); otherwise x as (K, M) box (64, 128), W as (N, K) box (64, 64).
constexpr int kMaxLinear = 3;
struct LinearMaps {
  CUtensorMap x[kMaxLinear];
  CUtensorMap w[kMaxLinear];
};
struct LinearProblem {
  const void *bias;  // [N] or nullptr
  void *y;           // [M, N]
  int M, N;
};
cudaError_t launch_linear_tc(const LinearMaps &maps, const LinearProblem *probs, int count,
                             int K, bool slabs, int *status, int num_sms, cudaStream_t stream);
// Slab tiling with every N >= 256: 128 x 256 tiles, stages of 64 of K; x's
// map then has box (64, 128, 1) and W's box (64, 64, 4)
bool linear_wide(int K, bool slabs, int min_n);

}  // namespace mha
