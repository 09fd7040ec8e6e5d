// attn_api.cu -- host side of the C ABI declared in include/attn.h:
// argument validation, per-device scratch (status word, internal block
// mask), option handling and the launches of the block-mask builder and the
// forward kernel.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "attn_internal.h"

namespace attn {
namespace {

struct Options {
  double rescale_threshold = 8.0;
  double force_partial = 0.0;
  double wait_budget_ms = 2000.0;
  double num_ctas = 0.0;
  double poly_fraction = 0.0;
  double debug_stall = 0.0;
};
Options g_opts;
std::mutex g_opts_mu;

Options options_snapshot() {
  std::lock_guard<std::mutex> lk(g_opts_mu);
  return g_opts;
}

// Per-device scratch owned by the library: the status word and the block
// mask built when the caller passes none.  Allocated on first need, grown
// when a larger problem arrives, kept until process exit.
struct DeviceScratch {
  DeviceStatus* status = nullptr;
  void* mask = nullptr;
  size_t mask_bytes = 0;
};
std::mutex g_scratch_mu;
std::vector<DeviceScratch> g_scratch;

attn_status scratch_for(int dev, DeviceScratch** out) {
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if ((int)g_scratch.size() <= dev) g_scratch.resize(dev + 1);
  DeviceScratch& s = g_scratch[dev];
  if (s.status == nullptr) {
    void* p = nullptr;
    if (cudaMalloc(&p, sizeof(DeviceStatus)) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemset(p, 0, sizeof(DeviceStatus)) != cudaSuccess) {
      cudaFree(p);
      return ATTN_ERR_CUDA;
    }
    s.status = static_cast<DeviceStatus*>(p);
  }
  *out = &s;
  return ATTN_OK;
}

attn_status ensure_mask_capacity(DeviceScratch* s, size_t bytes) {
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (s->mask_bytes >= bytes) return ATTN_OK;
  // The old buffer may still be read by work in flight on some stream.
  if (s->mask != nullptr) {
    if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
    cudaFree(s->mask);
    s->mask = nullptr;
    s->mask_bytes = 0;
  }
  size_t cap = align_up(bytes < (1u << 20) ? (1u << 20) : bytes, 1u << 20);
  if (cudaMalloc(&s->mask, cap) != cudaSuccess) return ATTN_ERR_CUDA;
  s->mask_bytes = cap;
  return ATTN_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Shape and mod checks shared by every entry point.
attn_status check_problem(int B, int H, int S_q, int S_k, const attn_mod_desc* mod) {
  if (B <= 0 || H <= 0 || S_q <= 0 || S_k <= 0) return ATTN_ERR_INVALID_ARG;
  if (S_q >= (1 << 30) || S_k >= (1 << 30)) return ATTN_ERR_INVALID_ARG;
  if (mod == nullptr) return ATTN_OK;
  if (mod->version != ATTN_MOD_DESC_VERSION) return ATTN_ERR_INVALID_ARG;
  const uint32_t known_mask =
      ATTN_MASK_CAUSAL | ATTN_MASK_WINDOW | ATTN_MASK_DOCUMENT | ATTN_MASK_PREFIX_LM;
  const uint32_t known_score = ATTN_SCORE_ALIBI | ATTN_SCORE_SOFTCAP;
  if ((mod->mask_flags & ~known_mask) || (mod->score_flags & ~known_score))
    return ATTN_ERR_INVALID_ARG;
  if (mod->q_offset <= -(1 << 30) || mod->q_offset >= (1 << 30)) return ATTN_ERR_INVALID_ARG;
  if ((mod->mask_flags & ATTN_MASK_WINDOW) && mod->window <= 0) return ATTN_ERR_INVALID_ARG;
  if (mod->mask_flags & ATTN_MASK_DOCUMENT) {
    if (mod->doc_ids == nullptr || !aligned(mod->doc_ids, 4)) return ATTN_ERR_INVALID_ARG;
    if (S_q != S_k) return ATTN_ERR_INVALID_ARG;
  }
  if ((mod->mask_flags & ATTN_MASK_PREFIX_LM) &&
      (mod->prefix_len == nullptr || !aligned(mod->prefix_len, 4)))
    return ATTN_ERR_INVALID_ARG;
  if ((mod->score_flags & ATTN_SCORE_SOFTCAP) && !(isfinite(mod->softcap) && mod->softcap > 0.f))
    return ATTN_ERR_INVALID_ARG;
  if ((mod->score_flags & ATTN_SCORE_ALIBI) && mod->alibi_slopes != nullptr &&
      !aligned(mod->alibi_slopes, 4))
    return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

MaskParams mask_params(int S_q, int S_k, const attn_mod_desc* mod) {
  MaskParams mp;
  memset(&mp, 0, sizeof(mp));
  mp.S_q = S_q;
  mp.S_k = S_k;
  if (mod != nullptr) {
    mp.flags = mod->mask_flags;
    mp.window = (mod->mask_flags & ATTN_MASK_WINDOW) ? mod->window : 0;
    mp.q_offset = mod->q_offset;
    mp.doc_ids = (mod->mask_flags & ATTN_MASK_DOCUMENT) ? mod->doc_ids : nullptr;
    mp.prefix_len = (mod->mask_flags & ATTN_MASK_PREFIX_LM) ? mod->prefix_len : nullptr;
  }
  return mp;
}

}  // namespace

// ---- scratch for attn_fwd_noalloc ----------------------------------------
// Some callers may not allocate device memory on the call path: code that
// runs while a stream is being captured into a CUDA graph, runtimes that own
// all device memory through their own pool or budget, and latency-critical
// paths that cannot take the device-wide synchronisation cudaMalloc/cudaFree
// may cause.  attn_fwd allocates its status word and grows its block-mask
// buffer on first need; attn_fwd_noalloc instead uses this fixed array,
// which every GPU that loads the library holds until the process exits.
// Layout: a DeviceStatus in the first kNoAllocStatusBytes, the block mask
// after it.  Host code must not pass the symbol itself to a kernel (on the
// host it names a stand-in, not device memory); the device address comes
// from cudaGetSymbolAddress, once per device.
namespace {
constexpr size_t kNoAllocStatusBytes = 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of g_noalloc_scratch on device `dev` (the current device).
attn_status noalloc_scratch(int dev, void** out) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return ATTN_ERR_CUDA;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return ATTN_OK;
}
}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

int attn_abi_version(void) { return ATTN_ABI_VERSION; }

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK:
      return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG:
      return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED:
      return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA:
      return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT:
      return "ATTN_ERR_TIMEOUT";
    case ATTN_ERR_DEVICE_CHECK:
      return "ATTN_ERR_DEVICE_CHECK";
  }
  return "ATTN_ERR_UNKNOWN";
}

attn_status attn_set_option(attn_option opt, double value) {
  if (!isfinite(value)) return ATTN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_opts_mu);
  switch (opt) {
    case ATTN_OPT_RESCALE_THRESHOLD:
      if (value < 0.0 || value > 64.0) return ATTN_ERR_INVALID_ARG;
      g_opts.rescale_threshold = value;
      return ATTN_OK;
    case ATTN_OPT_FORCE_PARTIAL:
      if (value != 0.0 && value != 1.0) return ATTN_ERR_INVALID_ARG;
      g_opts.force_partial = value;
      return ATTN_OK;
    case ATTN_OPT_WAIT_BUDGET_MS:
      if (value < 1.0 || value > 60000.0) return ATTN_ERR_INVALID_ARG;
      g_opts.wait_budget_ms = value;
      return ATTN_OK;
    case ATTN_OPT_NUM_CTAS:
      if (value < 0.0 || value > 65535.0 || value != floor(value)) return ATTN_ERR_INVALID_ARG;
      g_opts.num_ctas = value;
      return ATTN_OK;
    case ATTN_OPT_EXP_POLY_FRACTION:
      if (value < 0.0 || value > 1.0) return ATTN_ERR_INVALID_ARG;
      g_opts.poly_fraction = value;
      return ATTN_OK;
    case ATTN_OPT_DEBUG_STALL:
      if (value != 0.0 && value != 1.0) return ATTN_ERR_INVALID_ARG;
      g_opts.debug_stall = value;
      return ATTN_OK;
  }
  return ATTN_ERR_INVALID_ARG;
}

attn_status attn_get_option(attn_option opt, double* value) {
  if (value == nullptr) return ATTN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_opts_mu);
  switch (opt) {
    case ATTN_OPT_RESCALE_THRESHOLD:
      *value = g_opts.rescale_threshold;
      return ATTN_OK;
    case ATTN_OPT_FORCE_PARTIAL:
      *value = g_opts.force_partial;
      return ATTN_OK;
    case ATTN_OPT_WAIT_BUDGET_MS:
      *value = g_opts.wait_budget_ms;
      return ATTN_OK;
    case ATTN_OPT_NUM_CTAS:
      *value = g_opts.num_ctas;
      return ATTN_OK;
    case ATTN_OPT_EXP_POLY_FRACTION:
      *value = g_opts.poly_fraction;
      return ATTN_OK;
    case ATTN_OPT_DEBUG_STALL:
      *value = g_opts.debug_stall;
      return ATTN_OK;
  }
  return ATTN_ERR_INVALID_ARG;
}

size_t attn_block_mask_bytes(int B, int H, int S_q, int S_k, const attn_mod_desc* mod) {
  if (check_problem(B, H, S_q, S_k, mod) != ATTN_OK) return 0;
  return block_mask_geom(B, S_q, S_k, mod ? mod->mask_flags : 0u).total;
}

attn_status attn_build_block_mask(int B, int H, int S_q, int S_k, const attn_mod_desc* mod,
                                  void* dst, size_t bytes, attn_stream_t stream) {
  attn_status st = check_problem(B, H, S_q, S_k, mod);
  if (st != ATTN_OK) return st;
  if (dst == nullptr || !aligned(dst, 16)) return ATTN_ERR_INVALID_ARG;
  const size_t need = block_mask_geom(B, S_q, S_k, mod ? mod->mask_flags : 0u).total;
  if (bytes < need) return ATTN_ERR_INVALID_ARG;
  const Options o = options_snapshot();
  cudaError_t err = launch_build_block_mask(B, S_q, S_k, mask_params(S_q, S_k, mod),
                                            o.force_partial != 0.0 ? 1 : 0, dst,
                                            reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_block_mask_stats(const void* block_mask, size_t bytes, attn_stream_t stream,
                                  int64_t* n_entries, int64_t* n_full, int64_t* n_partial,
                                  int64_t* n_empty) {
  if (block_mask == nullptr || bytes < sizeof(BlockMaskHeader)) return ATTN_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
  BlockMaskHeader h;
  if (cudaMemcpy(&h, block_mask, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (h.magic != kBlockMaskMagic || h.version != kBlockMaskVersion || h.total_bytes > bytes)
    return ATTN_ERR_INVALID_ARG;
  std::vector<int32_t> cnt(h.n_entries);
  std::vector<uint32_t> list((size_t)h.n_entries * h.nK);
  const char* base = static_cast<const char*>(block_mask);
  if (cudaMemcpy(cnt.data(), base + h.cnt_off, sizeof(int32_t) * cnt.size(),
                 cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemcpy(list.data(), base + h.list_off, sizeof(uint32_t) * list.size(),
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  int64_t ent = 0, full = 0, part = 0, empty = 0;
  for (int e = 0; e < h.n_entries; ++e) {
    const int p = e % h.nP;
    for (int j = 0; j < cnt[e]; ++j) {
      const uint32_t x = list[(size_t)e * h.nK + j];
      ++ent;
      for (int t = 0; t < 2; ++t) {
        if (2 * p + t >= h.nQ) continue;
        const uint32_t c = entry_cls(x, t);
        full += c == kFull;
        part += c == kPartial;
      }
    }
  }
  // EMPTY = every (query tile, key tile) pair not FULL or PARTIAL
  empty = (int64_t)h.bm * h.nQ * h.nK - full - part;
  if (n_entries) *n_entries = ent;
  if (n_full) *n_full = full;
  if (n_partial) *n_partial = part;
  if (n_empty) *n_empty = empty;
  return ATTN_OK;
}

attn_status attn_get_device_status(attn_stream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  DeviceScratch* s = nullptr;
  attn_status st = scratch_for(dev, &s);
  if (st != ATTN_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  DeviceStatus h;
  if (cudaMemcpy(&h, s->status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (h.code != 0 && cudaMemset(s->status, 0, sizeof(DeviceStatus)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return static_cast<attn_status>(h.code);
}

attn_status attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                     int H, int H_kv, int S_q, int S_k, int D, float scale,
                     const attn_mod_desc* mod, attn_stream_t stream) {
  // ---- host-side validation: nothing is enqueued on failure ------------
  attn_status st = check_problem(B, H, S_q, S_k, mod);
  if (st != ATTN_OK) return st;
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr) return ATTN_ERR_INVALID_ARG;
  if (H_kv <= 0 || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (!(isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
    return ATTN_ERR_INVALID_ARG;
  if (lse != nullptr && !aligned(lse, 4)) return ATTN_ERR_INVALID_ARG;
  const size_t qb = (size_t)B * H * S_q * D * 2, kb = (size_t)B * H_kv * S_k * D * 2;
  if ((size_t)B * H > (size_t)INT32_MAX || (size_t)B * H_kv * (size_t)S_k > (size_t)INT32_MAX * 128)
    return ATTN_ERR_INVALID_ARG;
  if (overlaps(out, qb, q, qb) || overlaps(out, qb, k, kb) || overlaps(out, qb, v, kb))
    return ATTN_ERR_INVALID_ARG;
  if (lse != nullptr) {
    const size_t lb = (size_t)B * H * S_q * 4;
    if (overlaps(lse, lb, q, qb) || overlaps(lse, lb, k, kb) || overlaps(lse, lb, v, kb) ||
        overlaps(lse, lb, out, qb))
      return ATTN_ERR_INVALID_ARG;
  }
  const uint32_t mflags = mod ? mod->mask_flags : 0u;
  const BlockMaskGeom g = block_mask_geom(B, S_q, S_k, mflags);
  if (mod != nullptr && mod->block_mask != nullptr &&
      (!aligned(mod->block_mask, 16) || mod->block_mask_bytes < g.total))
    return ATTN_ERR_INVALID_ARG;

  // ---- device work -------------------------------------------------------
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  DeviceScratch* scr = nullptr;
  st = scratch_for(dev, &scr);
  if (st != ATTN_OK) return st;
  const Options o = options_snapshot();
  const MaskParams mp = mask_params(S_q, S_k, mod);

  const void* bmask = (mod != nullptr) ? mod->block_mask : nullptr;
  if (bmask == nullptr) {
    st = ensure_mask_capacity(scr, g.total);
    if (st != ATTN_OK) return st;
    if (launch_build_block_mask(B, S_q, S_k, mp, o.force_partial != 0.0 ? 1 : 0, scr->mask, s) !=
        cudaSuccess)
      return ATTN_ERR_CUDA;
    bmask = scr->mask;
  }

  FwdArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.H_kv = H_kv;
  a.S_q = S_q;
  a.S_k = S_k;
  a.D = D;
  a.scale = scale;
  a.mask = mp;
  a.score_flags = mod ? mod->score_flags : 0u;
  a.softcap = mod ? mod->softcap : 0.f;
  a.alibi_slopes = (mod && (mod->score_flags & ATTN_SCORE_ALIBI)) ? mod->alibi_slopes : nullptr;
  a.block_mask = bmask;
  a.n_entries = g.n_entries;
  a.bm = g.bm;
  a.nP = g.nP;
  a.status = scr->status;
  a.rescale_threshold = (float)o.rescale_threshold;
  a.wait_budget_ms = o.wait_budget_ms;
  a.num_ctas = (int)o.num_ctas;
  a.poly_fraction = (float)o.poly_fraction;
  a.debug_stall = o.debug_stall != 0.0 ? 1 : 0;
  return launch_attn_fwd(a, s) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out, float* lse,
                             int B, int H, int H_kv, int S_q, int S_k, int D, float scale,
                             const attn_mod_desc* mod, attn_stream_t stream) {
  // ---- host-side validation (same rules as attn_fwd) -----------------------
  attn_status st = check_problem(B, H, S_q, S_k, mod);
  if (st != ATTN_OK) return st;
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr) return ATTN_ERR_INVALID_ARG;
  if (H_kv <= 0 || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (!(isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
    return ATTN_ERR_INVALID_ARG;
  if (lse != nullptr && !aligned(lse, 4)) return ATTN_ERR_INVALID_ARG;
  const size_t qb = (size_t)B * H * S_q * D * 2, kb = (size_t)B * H_kv * S_k * D * 2;
  if ((size_t)B * H > (size_t)INT32_MAX || (size_t)B * H_kv * (size_t)S_k > (size_t)INT32_MAX * 128)
    return ATTN_ERR_INVALID_ARG;
  if (overlaps(out, qb, q, qb) || overlaps(out, qb, k, kb) || overlaps(out, qb, v, kb))
    return ATTN_ERR_INVALID_ARG;
  if (lse != nullptr) {
    const size_t lb = (size_t)B * H * S_q * 4;
    if (overlaps(lse, lb, q, qb) || overlaps(lse, lb, k, kb) || overlaps(lse, lb, v, kb) ||
        overlaps(lse, lb, out, qb))
      return ATTN_ERR_INVALID_ARG;
  }
  // The block mask is always built into the fixed scratch array.
  if (mod != nullptr && mod->block_mask != nullptr) return ATTN_ERR_INVALID_ARG;
  const uint32_t mflags = mod ? mod->mask_flags : 0u;
  const BlockMaskGeom g = block_mask_geom(B, S_q, S_k, mflags);
  if (g.total > ATTN_NOALLOC_SCRATCH_BYTES - kNoAllocStatusBytes) return ATTN_ERR_UNSUPPORTED;

  // ---- device work: no allocation from here on ----------------------------
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  void* scratch = nullptr;
  st = noalloc_scratch(dev, &scratch);
  if (st != ATTN_OK) return st;
  DeviceStatus* status = static_cast<DeviceStatus*>(scratch);
  void* bmask = static_cast<char*>(scratch) + kNoAllocStatusBytes;
  // The status word must start at zero; the block mask is rewritten whole.
  if (cudaMemsetAsync(status, 0, sizeof(DeviceStatus), s) != cudaSuccess) return ATTN_ERR_CUDA;
  const Options o = options_snapshot();
  const MaskParams mp = mask_params(S_q, S_k, mod);
  if (launch_build_block_mask(B, S_q, S_k, mp, o.force_partial != 0.0 ? 1 : 0, bmask, s) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;

  FwdArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.H_kv = H_kv;
  a.S_q = S_q;
  a.S_k = S_k;
  a.D = D;
  a.scale = scale;
  a.mask = mp;
  a.score_flags = mod ? mod->score_flags : 0u;
  a.softcap = mod ? mod->softcap : 0.f;
  a.alibi_slopes = (mod && (mod->score_flags & ATTN_SCORE_ALIBI)) ? mod->alibi_slopes : nullptr;
  a.block_mask = bmask;
  a.n_entries = g.n_entries;
  a.bm = g.bm;
  a.nP = g.nP;
  a.status = status;
  a.rescale_threshold = (float)o.rescale_threshold;
  a.wait_budget_ms = o.wait_budget_ms;
  a.num_ctas = (int)o.num_ctas;
  a.poly_fraction = (float)o.poly_fraction;
  a.debug_stall = o.debug_stall != 0.0 ? 1 : 0;
  return launch_attn_fwd(a, s) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // extern "C"
