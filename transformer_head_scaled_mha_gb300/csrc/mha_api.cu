// C ABI of the library: argument validation, path selection, TMA descriptor
// encoding and kernel launch on the caller's stream.  See include/mha.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/mha.h"
#include "common.cuh"

namespace mha {
namespace {

// Device status word: a kernel whose bounded wait gave up writes
// kStatusTimeout here.  One per device, in the module's static memory.
__device__ int g_status = 0;

// Wait limit and test stall handed to every kernel (mha_debug_set_wait).
std::atomic<unsigned long long> g_wait_ns{kWaitLimitNs};
std::atomic<int> g_stall{0};

enum Path { kPathNone = 0, kPathF32 = 1, kPathShort = 2, kPathLong = 3, kPathZero = 4, kPathDecode = 5 };

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];

int sm_count(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return 0;
  int v = g_sms[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  g_sms[dev].store(v, std::memory_order_relaxed);
  return v;
}

// ---- per-context caches ----------------------------------------------------
// Device addresses of the module's symbols, and whether a kernel's attributes
// were set, belong to a CUDA context: after a device reset (or in another
// context on the same device) the module is loaded again and its symbols may
// move.  Entries are therefore keyed by the context's process-unique id; a
// thread with no current context (id 0) gets no cached answer.
typedef CUresult (*PfnCtxGetCurrent)(CUcontext *);
typedef CUresult (*PfnCtxGetId)(CUcontext, unsigned long long *);
PfnCtxGetCurrent g_ctx_get_current = nullptr;
PfnCtxGetId g_ctx_get_id = nullptr;
std::once_flag g_ctx_once;

unsigned long long current_ctx_id() {
  std::call_once(g_ctx_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<PfnCtxGetCurrent>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_id = reinterpret_cast<PfnCtxGetId>(fn);
  });
  if (g_ctx_get_current == nullptr || g_ctx_get_id == nullptr) return 0;
  CUcontext c = nullptr;
  if (g_ctx_get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
  unsigned long long id = 0;
  if (g_ctx_get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// (context id, key) -> value, a small table searched under a lock; when full,
// the oldest entry is replaced
struct CtxEntry {
  unsigned long long ctx;
  const void *key;
  void *value;
};
constexpr int kCtxEntries = 256;
CtxEntry g_ctx_table[kCtxEntries];
int g_ctx_next = 0;
std::mutex g_ctx_mu;

bool ctx_lookup(unsigned long long ctx, const void *key, void **value) {
  if (ctx == 0) return false;
  std::lock_guard<std::mutex> lock(g_ctx_mu);
  for (const CtxEntry &e : g_ctx_table)
    if (e.ctx == ctx && e.key == key) {
      *value = e.value;
      return true;
    }
  return false;
}
void ctx_store(unsigned long long ctx, const void *key, void *value) {
  if (ctx == 0) return;
  std::lock_guard<std::mutex> lock(g_ctx_mu);
  for (CtxEntry &e : g_ctx_table)
    if (e.ctx == ctx && e.key == key) {
      e.value = value;
      return;
    }
  g_ctx_table[g_ctx_next] = CtxEntry{ctx, key, value};
  g_ctx_next = (g_ctx_next + 1) % kCtxEntries;
}

// Device address of a module symbol in the current context.
void *symbol_ptr(const void *symbol) {
  const unsigned long long ctx = current_ctx_id();
  void *v = nullptr;
  if (ctx_lookup(ctx, symbol, &v)) return v;
  if (cudaGetSymbolAddress(&v, symbol) != cudaSuccess) return nullptr;
  ctx_store(ctx, symbol, v);
  return v;
}

int *status_ptr() { return static_cast<int *>(symbol_ptr(reinterpret_cast<const void *>(&g_status))); }

}  // namespace

cudaError_t set_smem_once(const void *kernel, int bytes) {
  const unsigned long long ctx = current_ctx_id();
  void *v = nullptr;
  if (ctx_lookup(ctx, kernel, &v) && reinterpret_cast<intptr_t>(v) == bytes) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) ctx_store(ctx, kernel, reinterpret_cast<void *>(static_cast<intptr_t>(bytes)));
  return e;
}

namespace {

int next_pow2(int x) {
  int r = 1;
  while (r < x) r <<= 1;
  return r;
}

// 4-D view (d, L, heads, B) of a contiguous bf16 tensor in either layout,
// 128-byte swizzle; box (64, box_rows, box_heads, 1)
bool make_map(CUtensorMap *map, const void *base, int d, int L, int heads, int B, int layout,
              int box_rows, int box_heads) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t e = 2;  // bytes per element
  const cuuint64_t row = layout == kLayoutBHSD ? d * e : static_cast<cuuint64_t>(heads) * d * e;
  const cuuint64_t head = layout == kLayoutBHSD ? static_cast<cuuint64_t>(L) * d * e : d * e;
  const cuuint64_t batch = static_cast<cuuint64_t>(heads) * L * d * e;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(L),
                              static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {row, head, batch};
  const cuuint32_t box[4] = {64u, static_cast<cuuint32_t>(box_rows),
                             static_cast<cuuint32_t>(box_heads), 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D view (cols, rows) of a row-major bf16 matrix, 128-byte swizzle
bool make_map_2d(CUtensorMap *map, const void *base, int cols, int rows, int box_cols,
                 int box_rows) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D view (64, rows, cols / 64) of a row-major bf16 matrix whose column
// count is a multiple of 64: 64-wide column slabs, 128-byte swizzle; box
// (64, box_rows, box_slabs)
bool make_map_slabs(CUtensorMap *map, const void *base, int cols, int rows, int box_rows,
                    int box_slabs = 2) {
  auto enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(cols / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2, 128};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows),
                             static_cast<cuuint32_t>(box_slabs)};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Validates and picks a path; returns a non-negative Path or -(mha_status).
int select_path(int B, int H, int H_kv, int Lq, int Lk, int dk, int dv, int mask, int dtype) {
  if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || dk <= 0 || dv <= 0) return -MHA_ERR_INVALID_ARGUMENT;
  if (H_kv <= 0 ? H > 0 : (H % H_kv) != 0) return -MHA_ERR_INVALID_ARGUMENT;
  if (mask & ~(kMaskCausal | kMaskKeyPadding | kMaskQueryPadding | kMaskCausalTail))
    return -MHA_ERR_INVALID_ARGUMENT;
  if ((mask & kMaskCausalTail) && (mask & (kMaskCausal | kMaskQueryPadding)))
    return -MHA_ERR_INVALID_ARGUMENT;
  if ((mask & (kMaskCausal | kMaskQueryPadding)) && Lq != Lk) return -MHA_ERR_INVALID_ARGUMENT;
  if (dtype != MHA_DTYPE_F32 && dtype != MHA_DTYPE_BF16) return -MHA_ERR_INVALID_ARGUMENT;
  // TMA coordinates and the kernels' row indices are 32-bit
  if (static_cast<long long>(B) * H > 0x7fffffffLL) return -MHA_ERR_UNSUPPORTED;
  if (dtype == MHA_DTYPE_F32) {
    if (dk > 128 || dv > 128) return -MHA_ERR_UNSUPPORTED;
  } else {
    if (dk != dv || (dk != 64 && dk != 128)) return -MHA_ERR_UNSUPPORTED;
  }
  if (static_cast<long long>(B) * H * Lq == 0) return kPathNone;
  if (Lk == 0) return kPathZero;
  if (dtype == MHA_DTYPE_F32) return kPathF32;
  // a few query rows per key/value head (decoding steps): keys on the lanes
  const long long rows_per_kv = static_cast<long long>(H / H_kv) * Lq;
  if ((mask & ~(kMaskKeyPadding | kMaskCausalTail)) == 0 && rows_per_kv <= 16 &&
      (Lk > 128 || dk == 128))
    return kPathDecode;
  // the packed kernel's 32-bit row strides need H <= 2^24
  if (dk == 64 && Lq <= 128 && Lk <= 128 && H <= (1 << 24)) return kPathShort;
  return kPathLong;
}

}  // namespace
}  // namespace mha

using namespace mha;

extern "C" int mha_fwd_path(int B, int H, int Lq, int Lk, int d_k, int d_v, int mask_kind,
                            int dtype) {
  return select_path(B, H, H, Lq, Lk, d_k, d_v, mask_kind, dtype);
}

extern "C" int mha_fwd_path_ex(int B, int H, int H_kv, int Lq, int Lk, int d_k, int d_v,
                               int mask_kind, int dtype) {
  return select_path(B, H, H_kv, Lq, Lk, d_k, d_v, mask_kind, dtype);
}

namespace {

// mha_fwd_ex, and with `lse` non-null each row's statistics for the backward
int fwd_impl(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H,
             int H_kv, int Lq, int Lk, int d_k, int d_v, int layout, int mask_kind,
             const int32_t *key_lengths, float scale, int dtype, void *stream_) {
  const int path = select_path(B, H, H_kv, Lq, Lk, d_k, d_v, mask_kind, dtype);
  if (path < 0) return -path;
  if (layout != kLayoutBHSD && layout != kLayoutBSHD) return MHA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(scale)) return MHA_ERR_INVALID_ARGUMENT;
  if (path == kPathNone) return MHA_OK;
  const bool padded = (mask_kind & (kMaskKeyPadding | kMaskQueryPadding)) != 0;
  if (padded && (key_lengths == nullptr || reinterpret_cast<uintptr_t>(key_lengths) % 4 != 0))
    return MHA_ERR_INVALID_ARGUMENT;
  const size_t esz = dtype == MHA_DTYPE_F32 ? 4 : 2;
  const size_t nq = static_cast<size_t>(B) * H * Lq * d_k * esz;
  const size_t nk = static_cast<size_t>(B) * H_kv * Lk * d_k * esz;
  const size_t nv = static_cast<size_t>(B) * H_kv * Lk * d_v * esz;
  const size_t no = static_cast<size_t>(B) * H * Lq * d_v * esz;
  if (out == nullptr || q == nullptr || (Lk > 0 && (k == nullptr || v == nullptr)))
    return MHA_ERR_INVALID_ARGUMENT;
  for (const void *ptr : {static_cast<const void *>(q), static_cast<const void *>(k),
                          static_cast<const void *>(v), static_cast<const void *>(out)})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return MHA_ERR_INVALID_ARGUMENT;
  if (overlaps(out, no, q, nq) || overlaps(out, no, k, nk) || overlaps(out, no, v, nv) ||
      (padded && overlaps(out, no, key_lengths, sizeof(int32_t) * B)))
    return MHA_ERR_INVALID_ARGUMENT;
  const size_t nl = sizeof(float) * static_cast<size_t>(B) * H * Lq;
  if (lse != nullptr &&
      (reinterpret_cast<uintptr_t>(lse) % 4 != 0 || overlaps(lse, nl, out, no) ||
       overlaps(lse, nl, q, nq) || overlaps(lse, nl, k, nk) || overlaps(lse, nl, v, nv) ||
       (padded && overlaps(lse, nl, key_lengths, sizeof(int32_t) * B))))
    return MHA_ERR_INVALID_ARGUMENT;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MHA_ERR_CUDA;
  Problem p{};
  p.B = B;
  p.H = H;
  p.Hkv = H_kv;
  p.Lq = Lq;
  p.Lk = Lk;
  p.dk = d_k;
  p.dv = d_v;
  p.layout = layout;
  p.mask = mask_kind;
  p.key_lengths = padded ? key_lengths : nullptr;
  p.scale_log2 = scale * kLog2e;
  p.status = status_ptr();
  if (p.status == nullptr) return MHA_ERR_CUDA;
  p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  p.stall = g_stall.load(std::memory_order_relaxed);
  p.lse = lse;

  cudaError_t err = cudaSuccess;
  if (path == kPathZero) {
    // no keys: every row is stored as zeros and has no statistics
    err = launch_zero_fill(out, no, stream);
    if (err == cudaSuccess && lse != nullptr)
      err = launch_fill_f32(lse, nl / sizeof(float), INFINITY, stream);
  } else if (path == kPathF32) {
    err = launch_f32_simt(static_cast<const float *>(q), static_cast<const float *>(k),
                          static_cast<const float *>(v), static_cast<float *>(out), p, stream);
  } else {
    const int sms = sm_count(dev);
    if (sms <= 0) return MHA_ERR_CUDA;
    if (path == kPathShort) {
      ShortGeom g{};
      g.Rq = next_pow2(Lq < 8 ? 8 : Lq);
      g.Rk = next_pow2(Lk < 16 ? 16 : Lk);
      g.P = 128 / (g.Rq > g.Rk ? g.Rq : g.Rk);
      if (g.P > H) g.P = H;  // a unit holds heads of one batch element
      g.units_per_b = (H + g.P - 1) / g.P;
      if (static_cast<long long>(B) * g.units_per_b > 0x7fffffffLL) return MHA_ERR_UNSUPPORTED;
      g.units = B * g.units_per_b;
      g.rows_q = (mask_kind & kMaskQueryPadding) ? 1 : 0;
      g.rows_k = (mask_kind & kMaskKeyPadding) ? 1 : 0;
      g.q = q;
      g.k = k;
      g.v = v;
      ShortMaps m;
      std::memset(&m, 0, sizeof m);
      const bool shared_kv = H_kv != H;
      bool ok = make_map(&m.q_full, q, 64, Lq, H, B, layout, g.Rq, g.P);
      if (ok && !shared_kv)
        ok = make_map(&m.k_full, k, 64, Lk, H_kv, B, layout, g.Rk, g.P) &&
             make_map(&m.v_full, v, 64, Lk, H_kv, B, layout, g.Rk, g.P);
      if (ok && shared_kv)
        ok = make_map(&m.k_one, k, 64, Lk, H_kv, B, layout, g.Rk, 1) &&
             make_map(&m.v_one, v, 64, Lk, H_kv, B, layout, g.Rk, 1);
      // one row-box map per height 8, 16, ..., Rq (Rk) for the padded tensors
      if (ok && (mask_kind & kMaskCausal) && g.Rq == 128)
        ok = make_map(&m.q_blk32, q, 64, Lq, H, B, layout, 32, 1);
      for (int h = 0; ok && g.rows_q && h < g.Rq / 8; ++h)
        ok = make_map(&m.q_rows[h], q, 64, Lq, H, B, layout, 8 * (h + 1), 1);
      // key/value row boxes: all P pairs of a unit at once when the heads
      // are not shared (the kernel packs their rows back to back)
      const int kv_box_heads = shared_kv ? 1 : g.P;
      for (int h = 0; ok && g.rows_k && h < g.Rk / 8; ++h)
        ok = make_map(&m.k_rows[h], k, 64, Lk, H_kv, B, layout, 8 * (h + 1), kv_box_heads) &&
             make_map(&m.v_rows[h], v, 64, Lk, H_kv, B, layout, 8 * (h + 1), kv_box_heads);
      if (!ok) return MHA_ERR_CUDA;
      err = launch_short_tc(m, g, p, out, sms, stream);
    } else if (path == kPathDecode) {
      DecodeMaps m;
      std::memset(&m, 0, sizeof m);
      bool ok = make_map(&m.q, q, d_k, Lq, H, B, layout, Lq, H / H_kv) &&
                make_map(&m.k, k, d_k, Lk, H_kv, B, layout, 128, 1) &&
                make_map(&m.v, v, d_v, Lk, H_kv, B, layout, 128, 1);
      if (!ok) return MHA_ERR_CUDA;
      err = launch_decode_tc(m, p, out, sms, stream);
    } else {
      LongMaps m;
      std::memset(&m, 0, sizeof m);
      bool ok = make_map(&m.q, q, d_k, Lq, H, B, layout, 128, 1) &&
                make_map(&m.k, k, d_k, Lk, H_kv, B, layout, 128, 1) &&
                make_map(&m.v, v, d_v, Lk, H_kv, B, layout, 128, 1) &&
                make_map(&m.o, out, d_v, Lq, H, B, layout, 128, 1);
      if (!ok) return MHA_ERR_CUDA;
      err = launch_long_tc(m, p, sms, stream);
    }
  }
  return err == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

}  // namespace

extern "C" int mha_fwd_ex(const void *q, const void *k, const void *v, void *out, int B, int H,
                          int H_kv, int Lq, int Lk, int d_k, int d_v, int layout, int mask_kind,
                          const int32_t *key_lengths, float scale, int dtype, void *stream) {
  return fwd_impl(q, k, v, out, nullptr, B, H, H_kv, Lq, Lk, d_k, d_v, layout, mask_kind,
                  key_lengths, scale, dtype, stream);
}

extern "C" int mha_fwd_lse(const void *q, const void *k, const void *v, void *out, float *lse,
                           int B, int H, int H_kv, int Lq, int Lk, int d_k, int d_v, int layout,
                           int mask_kind, const int32_t *key_lengths, float scale, int dtype,
                           void *stream) {
  if (lse == nullptr && static_cast<long long>(B) * H * Lq > 0) return MHA_ERR_INVALID_ARGUMENT;
  return fwd_impl(q, k, v, out, lse, B, H, H_kv, Lq, Lk, d_k, d_v, layout, mask_kind,
                  key_lengths, scale, dtype, stream);
}

extern "C" int mha_fwd(const void *q, const void *k, const void *v, void *out, int B, int H,
                       int Lq, int Lk, int d_k, int d_v, int mask_kind,
                       const int32_t *key_lengths, float scale, int dtype, void *stream) {
  return mha_fwd_ex(q, k, v, out, B, H, H, Lq, Lk, d_k, d_v, kLayoutBHSD, mask_kind, key_lengths,
                    scale, dtype, stream);
}

namespace {

constexpr size_t kBwdAlign = 256;
size_t bwd_round(size_t n) { return (n + kBwdAlign - 1) / kBwdAlign * kBwdAlign; }

}  // namespace

extern "C" size_t mha_bwd_workspace_size(int B, int H, int Lq) {
  if (B <= 0 || H <= 0 || Lq <= 0) return 0;
  return 2 * bwd_round(static_cast<size_t>(B) * H * Lq * sizeof(float));
}

namespace {

// mha_bwd, and with `lse_in` non-null the forward's row statistics in place of
// a statistics pass
int bwd_impl(const void *q, const void *k, const void *v, const void *out, const void *dout,
             const float *lse_in, void *dq, void *dk, void *dv, int B, int H, int H_kv, int Lq,
             int Lk, int d_k, int d_v, int layout, int mask_kind, const int32_t *key_lengths,
             float scale, int dtype, void *workspace, size_t workspace_bytes, void *stream_) {
  const int path = select_path(B, H, H_kv, Lq, Lk, d_k, d_v, mask_kind, dtype);
  if (path < 0) return -path;
  if (layout != kLayoutBHSD && layout != kLayoutBSHD) return MHA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(scale)) return MHA_ERR_INVALID_ARGUMENT;
  const bool padded = (mask_kind & (kMaskKeyPadding | kMaskQueryPadding)) != 0;
  if (padded && B > 0 &&
      (key_lengths == nullptr || reinterpret_cast<uintptr_t>(key_lengths) % 4 != 0))
    return MHA_ERR_INVALID_ARGUMENT;
  const size_t esz = dtype == MHA_DTYPE_F32 ? 4 : 2;
  const size_t nq = static_cast<size_t>(B) * H * Lq * d_k * esz;
  const size_t nk = static_cast<size_t>(B) * H_kv * Lk * d_k * esz;
  const size_t nv = static_cast<size_t>(B) * H_kv * Lk * d_v * esz;
  const size_t no = static_cast<size_t>(B) * H * Lq * d_v * esz;
  const size_t nws = mha_bwd_workspace_size(B, H, Lq);
  if (nq == 0 && nk == 0) return MHA_OK;
  const void *ins[5] = {q, k, v, out, dout};
  const size_t in_n[5] = {nq, nk, nv, no, no};
  void *outs[3] = {dq, dk, dv};
  const size_t out_n[3] = {nq, nk, nv};
  for (int i = 0; i < 5; ++i)
    if (in_n[i] > 0 && (ins[i] == nullptr || reinterpret_cast<uintptr_t>(ins[i]) % 16 != 0))
      return MHA_ERR_INVALID_ARGUMENT;
  for (int i = 0; i < 3; ++i)
    if (out_n[i] > 0 && (outs[i] == nullptr || reinterpret_cast<uintptr_t>(outs[i]) % 16 != 0))
      return MHA_ERR_INVALID_ARGUMENT;
  if (nws > 0 && (workspace == nullptr || workspace_bytes < nws ||
                  reinterpret_cast<uintptr_t>(workspace) % kBwdAlign != 0))
    return MHA_ERR_INVALID_ARGUMENT;
  // the gradients overlap no input, each other, the workspace or the lengths
  for (int o = 0; o < 3; ++o) {
    for (int i = 0; i < 5; ++i)
      if (overlaps(outs[o], out_n[o], ins[i], in_n[i])) return MHA_ERR_INVALID_ARGUMENT;
    for (int o2 = o + 1; o2 < 3; ++o2)
      if (overlaps(outs[o], out_n[o], outs[o2], out_n[o2])) return MHA_ERR_INVALID_ARGUMENT;
    if (overlaps(outs[o], out_n[o], workspace, nws)) return MHA_ERR_INVALID_ARGUMENT;
    if (padded && overlaps(outs[o], out_n[o], key_lengths, sizeof(int32_t) * B))
      return MHA_ERR_INVALID_ARGUMENT;
  }
  for (int i = 0; i < 5; ++i)
    if (overlaps(workspace, nws, ins[i], in_n[i])) return MHA_ERR_INVALID_ARGUMENT;
  if (padded && overlaps(workspace, nws, key_lengths, sizeof(int32_t) * B))
    return MHA_ERR_INVALID_ARGUMENT;
  const size_t nl = sizeof(float) * static_cast<size_t>(B) * H * Lq;
  if (lse_in != nullptr) {
    if (reinterpret_cast<uintptr_t>(lse_in) % 4 != 0 || overlaps(lse_in, nl, workspace, nws))
      return MHA_ERR_INVALID_ARGUMENT;
    for (int o = 0; o < 3; ++o)
      if (overlaps(outs[o], out_n[o], lse_in, nl)) return MHA_ERR_INVALID_ARGUMENT;
  }

  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MHA_ERR_CUDA;
  Problem p{};
  p.B = B;
  p.H = H;
  p.Hkv = H_kv;
  p.Lq = Lq;
  p.Lk = Lk;
  p.dk = d_k;
  p.dv = d_v;
  p.layout = layout;
  p.mask = mask_kind;
  p.key_lengths = padded ? key_lengths : nullptr;
  p.scale_log2 = scale * kLog2e;
  p.status = status_ptr();
  if (p.status == nullptr) return MHA_ERR_CUDA;
  p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  p.stall = g_stall.load(std::memory_order_relaxed);
  cudaError_t err = cudaSuccess;
  if (Lk == 0 || nq == 0) {
    // no keys: nothing reads q, k or v; every gradient is zero
    for (int i = 0; i < 3 && err == cudaSuccess; ++i)
      if (out_n[i] > 0) err = launch_zero_fill(outs[i], out_n[i], stream);
    return err == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
  }
  BwdArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.dout = dout;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  a.lse = reinterpret_cast<float *>(ws);
  a.dsum = reinterpret_cast<float *>(ws + nws / 2);
  a.scale = scale;
  a.pack = 1;
  if (dtype == MHA_DTYPE_BF16) {
    // tensor cores (d in {64, 128}, enforced by select_path).  The fused
    // short kernel packs pack = 128 / R pairs (R: the longer length rounded
    // up to a power of two) into one 128-row tile when the key/value heads
    // are not shared
    if (d_k == 64 && Lq <= 128 && Lk <= 128 && H_kv == H) {
      const int R = next_pow2(std::max(std::max(Lq, Lk), 8));
      a.pack = 128 / R;
      while (a.pack > 1 && a.pack > H) a.pack >>= 1;
    }
    const int rows = 128 / a.pack;
    LongMaps m;
    std::memset(&m, 0, sizeof m);
    const bool ok = make_map(&m.q, q, d_k, Lq, H, B, layout, rows, a.pack) &&
                    make_map(&m.k, k, d_k, Lk, H_kv, B, layout, rows, a.pack) &&
                    make_map(&m.v, v, d_v, Lk, H_kv, B, layout, rows, a.pack) &&
                    make_map(&m.o, dout, d_v, Lq, H, B, layout, rows, a.pack);
    if (!ok) return MHA_ERR_CUDA;
    const int sms = sm_count(dev);
    if (sms <= 0) return MHA_ERR_CUDA;
    if (lse_in != nullptr) a.lse = const_cast<float *>(lse_in);  // read only
    err = launch_bwd_tc(m, p, a, sms, stream, lse_in != nullptr);
  } else {
    // the fp32 path recomputes the statistics (its lse and D come together)
    err = launch_bwd_simt(a, p, false, stream);
  }
  return err == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

}  // namespace

extern "C" int mha_bwd(const void *q, const void *k, const void *v, const void *out,
                       const void *dout, void *dq, void *dk, void *dv, int B, int H, int H_kv,
                       int Lq, int Lk, int d_k, int d_v, int layout, int mask_kind,
                       const int32_t *key_lengths, float scale, int dtype, void *workspace,
                       size_t workspace_bytes, void *stream) {
  return bwd_impl(q, k, v, out, dout, nullptr, dq, dk, dv, B, H, H_kv, Lq, Lk, d_k, d_v, layout,
                  mask_kind, key_lengths, scale, dtype, workspace, workspace_bytes, stream);
}

extern "C" int mha_bwd_lse(const void *q, const void *k, const void *v, const void *out,
                           const void *dout, const float *lse, void *dq, void *dk, void *dv, int B,
                           int H, int H_kv, int Lq, int Lk, int d_k, int d_v, int layout,
                           int mask_kind, const int32_t *key_lengths, float scale, int dtype,
                           void *workspace, size_t workspace_bytes, void *stream) {
  if (lse == nullptr && static_cast<long long>(B) * H * Lq > 0) return MHA_ERR_INVALID_ARGUMENT;
  return bwd_impl(q, k, v, out, dout, lse, dq, dk, dv, B, H, H_kv, Lq, Lk, d_k, d_v, layout,
                  mask_kind, key_lengths, scale, dtype, workspace, workspace_bytes, stream);
}

namespace {

// Validation shared by mha_linear_fwd and the sublayer's projections.
int check_linear(const void *x, const void *w, const void *b, const void *y, long long M, int K,
                 int N, int dtype) {
  if (M < 0 || K <= 0 || N <= 0) return MHA_ERR_INVALID_ARGUMENT;
  if (dtype != MHA_DTYPE_F32 && dtype != MHA_DTYPE_BF16) return MHA_ERR_INVALID_ARGUMENT;
  if (dtype != MHA_DTYPE_BF16) return MHA_ERR_UNSUPPORTED;
  // the copy engine needs 16-byte row strides
  if (K % 8 != 0 || N % 8 != 0) return MHA_ERR_UNSUPPORTED;
  if (M > 0x7fffffffLL) return MHA_ERR_UNSUPPORTED;
  if (M == 0) return MHA_OK;
  if (x == nullptr || w == nullptr || y == nullptr) return MHA_ERR_INVALID_ARGUMENT;
  for (const void *ptr : {x, w, y})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return MHA_ERR_INVALID_ARGUMENT;
  if (b != nullptr && reinterpret_cast<uintptr_t>(b) % 2 != 0) return MHA_ERR_INVALID_ARGUMENT;
  const size_t ny = static_cast<size_t>(M) * N * 2;
  if (overlaps(y, ny, x, static_cast<size_t>(M) * K * 2) ||
      overlaps(y, ny, w, static_cast<size_t>(K) * N * 2) || overlaps(y, ny, b, N * 2))
    return MHA_ERR_INVALID_ARGUMENT;
  return MHA_OK;
}

// One validated product y = x W + b of a launch (M > 0).
struct LinearJob {
  const void *x, *w, *b;
  void *y;
  int M, N;
};

// One launch for up to kMaxLinear validated products with the same K.
int run_linears(const LinearJob *jobs, int count, int K, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MHA_ERR_CUDA;
  const int sms = sm_count(dev);
  int *status = status_ptr();
  if (sms <= 0 || status == nullptr) return MHA_ERR_CUDA;
  bool slabs = K % 64 == 0;
  for (int g = 0; g < count; ++g) slabs = slabs && jobs[g].N % 64 == 0;
  int min_n = jobs[0].N;
  for (int g = 1; g < count; ++g) min_n = std::min(min_n, jobs[g].N);
  const bool wide = linear_wide(K, slabs, min_n);
  LinearMaps m;
  std::memset(&m, 0, sizeof m);
  LinearProblem probs[kMaxLinear];
  for (int g = 0; g < count; ++g) {
    const LinearJob &j = jobs[g];
    const bool ok = slabs ? make_map_slabs(&m.x[g], j.x, K, j.M, 128, wide ? 1 : 2) &&
                                make_map_slabs(&m.w[g], j.w, j.N, K, wide ? 64 : 128,
                                               wide ? 4 : 2)
                          : make_map_2d(&m.x[g], j.x, K, j.M, 64, 128) &&
                                make_map_2d(&m.w[g], j.w, j.N, K, 64, 64);
    if (!ok) return MHA_ERR_CUDA;
    probs[g] = LinearProblem{j.b, j.y, j.M, j.N};
  }
  return launch_linear_tc(m, probs, count, K, slabs, status, sms, stream) == cudaSuccess
             ? MHA_OK
             : MHA_ERR_CUDA;
}

int run_linear(const void *x, const void *w, const void *b, void *y, int M, int K, int N,
               cudaStream_t stream) {
  const LinearJob j{x, w, b, y, M, N};
  return run_linears(&j, 1, K, stream);
}

constexpr size_t kWsAlign = 256;
size_t ws_round(size_t n) { return (n + kWsAlign - 1) / kWsAlign * kWsAlign; }

// Byte offsets of q, k, v and the concatenated heads in a sublayer workspace.
struct SublayerWs {
  size_t q, k, v, heads, total;
};
SublayerWs sublayer_ws(long long B, long long T, long long S, long long H, long long H_kv,
                       long long d_k, long long d_v) {
  SublayerWs w;
  w.q = 0;
  w.k = w.q + ws_round(static_cast<size_t>(B * T * H * d_k * 2));
  w.v = w.k + ws_round(static_cast<size_t>(B * S * H_kv * d_k * 2));
  w.heads = w.v + ws_round(static_cast<size_t>(B * S * H_kv * d_v * 2));
  w.total = w.heads + ws_round(static_cast<size_t>(B * T * H * d_v * 2));
  return w;
}

}  // namespace

extern "C" int mha_linear_fwd(const void *x, const void *w, const void *b, void *y, int M, int K,
                              int N, int dtype, void *stream) {
  const int st = check_linear(x, w, b, y, M, K, N, dtype);
  if (st != MHA_OK || M == 0) return st;
  return run_linear(x, w, b, y, M, K, N, static_cast<cudaStream_t>(stream));
}

extern "C" size_t mha_sublayer_workspace_size(int B, int T, int S, int d_model, int H, int H_kv,
                                              int d_k, int d_v) {
  (void)d_model;
  if (B < 0 || T < 0 || S < 0 || H < 0 || H_kv < 0 || d_k < 0 || d_v < 0) return 0;
  return sublayer_ws(B, T, S, H, H_kv, d_k, d_v).total;
}

extern "C" int mha_sublayer_fwd(const void *x, const void *mem, void *out, const void *w_q,
                                const void *w_k, const void *w_v, const void *w_o,
                                const void *b_q, const void *b_k, const void *b_v,
                                const void *b_o, int B, int T, int S, int d_model, int H,
                                int H_kv, int d_k, int d_v, int mask_kind,
                                const int32_t *key_lengths, float scale, int dtype,
                                void *workspace, size_t workspace_bytes, void *stream_) {
  if (mem == nullptr) {  // self-attention: keys and values come from x
    mem = x;
    if (S != T) return MHA_ERR_INVALID_ARGUMENT;
  }
  if (B < 0 || T < 0 || S < 0 || d_model <= 0 || H <= 0 || H_kv <= 0 || d_k <= 0 || d_v <= 0)
    return MHA_ERR_INVALID_ARGUMENT;
  if (H % H_kv != 0) return MHA_ERR_INVALID_ARGUMENT;
  const long long Mq = static_cast<long long>(B) * T, Mk = static_cast<long long>(B) * S;
  // every step's shape rules, before anything is enqueued
  int st;
  const SublayerWs ws = sublayer_ws(B, T, S, H, H_kv, d_k, d_v);
  uint8_t *wsb = static_cast<uint8_t *>(workspace);
  void *q = wsb + ws.q, *k = wsb + ws.k, *v = wsb + ws.v, *heads = wsb + ws.heads;
  // projection widths in 64 bits: a product past INT_MAX would otherwise wrap
  // to a small, valid-looking width
  const long long nq = static_cast<long long>(H) * d_k, nk = static_cast<long long>(H_kv) * d_k;
  const long long nv = static_cast<long long>(H_kv) * d_v, no = static_cast<long long>(H) * d_v;
  if (nq > 0x7fffffffLL || nk > 0x7fffffffLL || nv > 0x7fffffffLL || no > 0x7fffffffLL)
    return MHA_ERR_UNSUPPORTED;
  if ((st = check_linear(x, w_q, b_q, out, Mq, d_model, static_cast<int>(nq), dtype)) != MHA_OK ||
      (st = check_linear(mem, w_k, b_k, out, Mk, d_model, static_cast<int>(nk), dtype)) != MHA_OK ||
      (st = check_linear(mem, w_v, b_v, out, Mk, d_model, static_cast<int>(nv), dtype)) != MHA_OK ||
      (st = check_linear(heads, w_o, b_o, out, Mq, static_cast<int>(no), d_model, dtype)) != MHA_OK)
    return st;
  const int path = select_path(B, H, H_kv, T, S, d_k, d_v, mask_kind, dtype);
  if (path < 0) return -path;
  if (!std::isfinite(scale)) return MHA_ERR_INVALID_ARGUMENT;
  if (Mq == 0) return MHA_OK;
  const bool padded = (mask_kind & (kMaskKeyPadding | kMaskQueryPadding)) != 0;
  if (padded && (key_lengths == nullptr || reinterpret_cast<uintptr_t>(key_lengths) % 4 != 0))
    return MHA_ERR_INVALID_ARGUMENT;
  if (workspace == nullptr || workspace_bytes < ws.total ||
      reinterpret_cast<uintptr_t>(workspace) % kWsAlign != 0)
    return MHA_ERR_INVALID_ARGUMENT;
  const size_t n_out = static_cast<size_t>(Mq) * d_model * 2;
  if (overlaps(workspace, ws.total, out, n_out) ||
      overlaps(workspace, ws.total, x, static_cast<size_t>(Mq) * d_model * 2) ||
      overlaps(workspace, ws.total, mem, static_cast<size_t>(Mk) * d_model * 2) ||
      (padded && (overlaps(workspace, ws.total, key_lengths, sizeof(int32_t) * B) ||
                  overlaps(out, n_out, key_lengths, sizeof(int32_t) * B))))
    return MHA_ERR_INVALID_ARGUMENT;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  // 1. the three projections in one launch (head i of each is columns
  //    [i d, (i + 1) d): [B, L, heads, d])
  const LinearJob proj[3] = {
      {x, w_q, b_q, q, static_cast<int>(Mq), static_cast<int>(nq)},
      {mem, w_k, b_k, k, static_cast<int>(Mk), static_cast<int>(nk)},
      {mem, w_v, b_v, v, static_cast<int>(Mk), static_cast<int>(nv)}};
  if ((st = run_linears(proj, Mk > 0 ? 3 : 1, d_model, stream)) != MHA_OK) return st;
  // 2. attention per head, in the [B, L, heads, d] layout
  if ((st = mha_fwd_ex(q, k, v, heads, B, H, H_kv, T, S, d_k, d_v, kLayoutBSHD, mask_kind,
                       key_lengths, scale, dtype, stream)) != MHA_OK)
    return st;
  // 3. concatenated heads [B, T, H d_v] times W_o
  return run_linear(heads, w_o, b_o, out, static_cast<int>(Mq), static_cast<int>(no), d_model, stream);
}

namespace {

// Scratch for mha_sublayer_fwd_static: the library's own device memory for the
// projected q, k, v and the concatenated heads, a fixed 64 MiB per device
// (enough for the Transformer-base encoder sublayer at B = 256, T = 64,
// d_model = 512).  It is reserved when the module is loaded, never by a call.
constexpr size_t kStaticScratchBytes = static_cast<size_t>(64) << 20;
__device__ __align__(256) uint8_t g_sublayer_scratch[kStaticScratchBytes];

// Device address of the current device's scratch: a symbol lookup
// (cudaGetSymbolAddress, not an allocation), made by the first call in each
// CUDA context and cached for that context; the host-side name of the array
// is only a stand-in and is never handed to a kernel.
void *scratch_ptr() {
  return symbol_ptr(reinterpret_cast<const void *>(&g_sublayer_scratch[0]));
}

}  // namespace

// For callers that cannot hand the sublayer a workspace: hosts whose device
// memory is budgeted up front and that must not allocate on their serving
// path, or C callers without a device allocator of their own.  Same
// computation as mha_sublayer_fwd, with the library's static scratch as the
// workspace; no allocation and no allocating library call.  Nothing in the
// scratch must start at zero: every step writes its output in full before the
// next reads it.  All calls on a device share the one scratch, so calls that
// overlap in time (other streams, other threads) race on it.
extern "C" int mha_sublayer_fwd_static(const void *x, const void *mem, void *out,
                                       const void *w_q, const void *w_k, const void *w_v,
                                       const void *w_o, const void *b_q, const void *b_k,
                                       const void *b_v, const void *b_o, int B, int T, int S,
                                       int d_model, int H, int H_kv, int d_k, int d_v,
                                       int mask_kind, const int32_t *key_lengths, float scale,
                                       int dtype, void *stream) {
  if (B < 0 || T < 0 || S < 0 || H < 0 || H_kv < 0 || d_k < 0 || d_v < 0)
    return MHA_ERR_INVALID_ARGUMENT;
  if (sublayer_ws(B, T, S, H, H_kv, d_k, d_v).total > kStaticScratchBytes)
    return MHA_ERR_UNSUPPORTED;  // larger than the static scratch: use mha_sublayer_fwd
  if (static_cast<long long>(B) * T == 0)
    return mha_sublayer_fwd(x, mem, out, w_q, w_k, w_v, w_o, b_q, b_k, b_v, b_o, B, T, S,
                            d_model, H, H_kv, d_k, d_v, mask_kind, key_lengths, scale, dtype,
                            nullptr, 0, stream);
  void *scratch = scratch_ptr();
  if (scratch == nullptr) return MHA_ERR_CUDA;
  return mha_sublayer_fwd(x, mem, out, w_q, w_k, w_v, w_o, b_q, b_k, b_v, b_o, B, T, S, d_model,
                          H, H_kv, d_k, d_v, mask_kind, key_lengths, scale, dtype, scratch,
                          kStaticScratchBytes, stream);
}

extern "C" const char *mha_status_string(int status) {
  switch (status) {
    case MHA_OK: return "ok";
    case MHA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case MHA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case MHA_ERR_CUDA: return "CUDA error";
    case MHA_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

extern "C" int mha_debug_status(void *stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int host = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbolAsync(&host, g_status, sizeof(int), 0, cudaMemcpyDeviceToHost,
                                stream) != cudaSuccess)
    return MHA_ERR_CUDA;
  if (cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream) !=
      cudaSuccess)
    return MHA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MHA_ERR_CUDA;
  return host == 0 ? MHA_OK : MHA_ERR_TIMEOUT;
}

extern "C" int mha_debug_set_wait(unsigned long long limit_ns, int stall) {
  if (stall & ~(kStallShortMma | kStallLongMma)) return MHA_ERR_INVALID_ARGUMENT;
  g_wait_ns.store(limit_ns == 0 ? kWaitLimitNs : limit_ns, std::memory_order_relaxed);
  g_stall.store(stall, std::memory_order_relaxed);
  return MHA_OK;
}

extern "C" int mha_version(void) { return 100; }
