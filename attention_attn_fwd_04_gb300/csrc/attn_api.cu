// attn_api.cu -- host side of the C ABI declared in include/attn.h:
// argument validation, per-device scratch (status word, internal block
// mask), option handling and the launches of the block-mask builder and the
// forward kernel.
#include <cuda_runtime.h>
#include <math.h>
#include <stddef.h>
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
  double cta_pair = 0.0;
};
Options g_opts;
std::mutex g_opts_mu;

Options options_snapshot() {
  std::lock_guard<std::mutex> lk(g_opts_mu);
  return g_opts;
}

// Query tiles per entry of the forward's block masks under these options.
int mask_tpe(const Options& o) { return o.cta_pair != 0.0 ? kTilesPerQuad : kTilesPerItem; }

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

// Per-device scratch of attn_bwd: its own block masks (forward and
// transposed) and the row statistics, grown on demand like the forward's.
struct BwdScratch {
  void* buf = nullptr;
  size_t bytes = 0;
};
std::mutex g_bwd_mu;
std::vector<BwdScratch> g_bwd;

attn_status bwd_scratch(int dev, size_t bytes, void** out) {
  std::lock_guard<std::mutex> lk(g_bwd_mu);
  if ((int)g_bwd.size() <= dev) g_bwd.resize(dev + 1);
  BwdScratch& s = g_bwd[dev];
  if (s.bytes < bytes) {
    if (s.buf != nullptr) {
      if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
      cudaFree(s.buf);
      s.buf = nullptr;
      s.bytes = 0;
    }
    const size_t cap = align_up(bytes, 1u << 20);
    if (cudaMalloc(&s.buf, cap) != cudaSuccess) {
      s.buf = nullptr;
      return ATTN_ERR_CUDA;
    }
    s.bytes = cap;
  }
  *out = s.buf;
  return ATTN_OK;
}

// A caller's descriptor as the current layout: a version-1 descriptor is
// copied up to its end (it has no version-2 fields) and the rest zeroed.
// Returns nullptr for no descriptor; *st is INVALID_ARG for an unknown
// version.
const attn_mod_desc* load_mod(const attn_mod_desc* in, attn_mod_desc* buf, attn_status* st) {
  *st = ATTN_OK;
  if (in == nullptr) return nullptr;
  memset(buf, 0, sizeof(*buf));
  if (in->version == 1u) {
    memcpy(buf, in, offsetof(attn_mod_desc, blocks));
  } else if (in->version == ATTN_MOD_DESC_VERSION) {
    *buf = *in;
  } else {
    *st = ATTN_ERR_INVALID_ARG;
    return nullptr;
  }
  buf->version = ATTN_MOD_DESC_VERSION;
  return buf;
}

// The mask flags the kernels see: the caller's, plus the internal bit
// that makes the block mask per batch entry for a per-batch block map.
uint32_t kernel_mask_flags(const attn_mod_desc* mod) {
  if (mod == nullptr) return 0u;
  uint32_t f = mod->mask_flags;
  if ((f & ATTN_MASK_BLOCKS) && mod->blocks_batched) f |= kMaskBlocksBatched;
  return f;
}

// Shape and mod checks shared by every entry point (on a loaded descriptor).
attn_status check_problem(int B, int H, int S_q, int S_k, const attn_mod_desc* mod) {
  if (B <= 0 || H <= 0 || S_q <= 0 || S_k <= 0) return ATTN_ERR_INVALID_ARG;
  if (S_q >= (1 << 30) || S_k >= (1 << 30)) return ATTN_ERR_INVALID_ARG;
  if (mod == nullptr) return ATTN_OK;
  if (mod->version != ATTN_MOD_DESC_VERSION) return ATTN_ERR_INVALID_ARG;
  const uint32_t known_mask = ATTN_MASK_CAUSAL | ATTN_MASK_WINDOW | ATTN_MASK_DOCUMENT |
                              ATTN_MASK_PREFIX_LM | ATTN_MASK_BLOCKS;
  const uint32_t known_score = ATTN_SCORE_ALIBI | ATTN_SCORE_SOFTCAP | ATTN_SCORE_RELBIAS;
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
  if ((mod->mask_flags & ATTN_MASK_BLOCKS) &&
      (mod->blocks == nullptr || (mod->blocks_batched != 0 && mod->blocks_batched != 1)))
    return ATTN_ERR_INVALID_ARG;
  if ((mod->score_flags & ATTN_SCORE_RELBIAS) &&
      (mod->rel_bias == nullptr || !aligned(mod->rel_bias, 4) || mod->rel_max < 0 ||
       mod->rel_max >= (1 << 30)))
    return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

MaskParams mask_params(int S_q, int S_k, const attn_mod_desc* mod) {
  MaskParams mp;
  memset(&mp, 0, sizeof(mp));
  mp.S_q = S_q;
  mp.S_k = S_k;
  if (mod != nullptr) {
    mp.flags = kernel_mask_flags(mod);
    mp.window = (mod->mask_flags & ATTN_MASK_WINDOW) ? mod->window : 0;
    mp.q_offset = mod->q_offset;
    mp.doc_ids = (mod->mask_flags & ATTN_MASK_DOCUMENT) ? mod->doc_ids : nullptr;
    mp.prefix_len = (mod->mask_flags & ATTN_MASK_PREFIX_LM) ? mod->prefix_len : nullptr;
    mp.blocks = (mod->mask_flags & ATTN_MASK_BLOCKS) ? mod->blocks : nullptr;
  }
  return mp;
}

// Checks on the tensors of one forward that do not depend on where they
// live: present, head grouping, scale, head dim, sizes that index in 32
// bits, outputs not overlapping inputs.
attn_status check_tensors(const void* q, const void* k, const void* v, const void* out,
                          const float* lse, int B, int H, int H_kv, int S_q, int S_k, int D,
                          float scale) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr) return ATTN_ERR_INVALID_ARG;
  if (H_kv <= 0 || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (!(isfinite(scale) && scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if ((size_t)B * H > (size_t)INT32_MAX || (size_t)B * H_kv * (size_t)S_k > (size_t)INT32_MAX * 128)
    return ATTN_ERR_INVALID_ARG;
  const size_t qb = (size_t)B * H * S_q * D * 2, kb = (size_t)B * H_kv * S_k * D * 2;
  if (overlaps(out, qb, q, qb) || overlaps(out, qb, k, kb) || overlaps(out, qb, v, kb))
    return ATTN_ERR_INVALID_ARG;
  if (lse != nullptr) {
    const size_t lb = (size_t)B * H * S_q * 4;
    if (overlaps(lse, lb, q, qb) || overlaps(lse, lb, k, kb) || overlaps(lse, lb, v, kb) ||
        overlaps(lse, lb, out, qb))
      return ATTN_ERR_INVALID_ARG;
  }
  return ATTN_OK;
}

// Device tensors additionally need 16-byte (Q, K, V, O) and 4-byte (LSE)
// alignment for the tensor maps and the vector stores.
attn_status check_device_tensors(const void* q, const void* k, const void* v, const void* out,
                                 const float* lse, int B, int H, int H_kv, int S_q, int S_k,
                                 int D, float scale) {
  attn_status st = check_tensors(q, k, v, out, lse, B, H, H_kv, S_q, S_k, D, scale);
  if (st != ATTN_OK) return st;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
    return ATTN_ERR_INVALID_ARG;
  if (lse != nullptr && !aligned(lse, 4)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

// Enqueues one checked forward on s: the block-mask build into mask_buf
// (skipped when bmask is given) and the forward kernel.
attn_status enqueue_forward(const void* q, const void* k, const void* v, void* out, float* lse,
                            int B, int H, int H_kv, int S_q, int S_k, int D, float scale,
                            const attn_mod_desc* mod, const void* bmask, void* mask_buf,
                            DeviceStatus* status, const Options& o, cudaStream_t s) {
  const MaskParams mp = mask_params(S_q, S_k, mod);
  const int tpe = mask_tpe(o);
  const BlockMaskGeom g = block_mask_geom(B, S_q, S_k, mp.flags, tpe);
  if (bmask == nullptr) {
    if (launch_build_block_mask(B, S_q, S_k, mp, o.force_partial != 0.0 ? 1 : 0, mask_buf, s,
                                tpe) != cudaSuccess)
      return ATTN_ERR_CUDA;
    bmask = mask_buf;
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
  if (mod && (mod->score_flags & ATTN_SCORE_RELBIAS)) {
    a.rel_bias = mod->rel_bias;
    a.rel_max = mod->rel_max;
  }
  a.block_mask = bmask;
  a.n_entries = g.n_entries;
  a.bm = g.bm;
  a.nP = g.nP;
  a.status = status;
  a.rescale_threshold = (float)o.rescale_threshold;
  a.wait_budget_ms = o.wait_budget_ms;
  a.num_ctas = (int)o.num_ctas;
  a.cta_pair = o.cta_pair != 0.0 ? 1 : 0;
  a.tpe = tpe;
  a.poly_fraction = (float)o.poly_fraction;
  a.debug_stall = o.debug_stall != 0.0 ? 1 : 0;
  return launch_attn_fwd(a, s) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
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
constexpr size_t kNoAllocStatusBytes = ATTN_NOALLOC_STATUS_BYTES;
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

// ---- pipeline for attn_fwd_host -------------------------------------------
// Host-memory callers pay for the copies in and out.  Each device gets three
// streams of the library's own -- host-to-device copies, compute,
// device-to-host copies -- and two slots of device memory used by
// alternate calls, so one call's input copy runs while the previous call
// computes and the one before copies its results out.  Every hand-over is
// an event: a slot is refilled only after its previous results have left.
struct HostSlot {
  void* buf = nullptr;
  size_t bytes = 0;
  cudaEvent_t done = nullptr;  // the slot's last output copy
  bool used = false;
};
struct HostPipe {
  std::mutex mu;
  bool ready = false;
  cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
  // hand-overs; each wait is enqueued before the event is recorded again
  cudaEvent_t user = nullptr, in = nullptr, comp_ev = nullptr;
  HostSlot slot[2];
  int next = 0;
};
constexpr int kHostChunks = 8;
constexpr int kHostMaxDevices = 64;
std::mutex g_host_mu;
HostPipe g_host[kHostMaxDevices];

attn_status host_pipe(int dev, HostPipe** out) {
  if (dev < 0 || dev >= kHostMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_host_mu);
  HostPipe& p = g_host[dev];
  if (!p.ready) {
    const unsigned fl = cudaStreamNonBlocking;
    const unsigned ev = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&p.h2d, fl) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.comp, fl) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.d2h, fl) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.user, ev) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.in, ev) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.comp_ev, ev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    for (HostSlot& sl : p.slot)
      if (cudaEventCreateWithFlags(&sl.done, ev) != cudaSuccess) return ATTN_ERR_CUDA;
    p.ready = true;
  }
  *out = &p;
  return ATTN_OK;
}

// Byte offsets of one call's device copies inside a slot.
struct HostLayout {
  size_t q, k, v, o, lse, doc, prefix, slopes, blocks, rel, mask, total;
  size_t blocks_bytes, rel_bytes;
};
HostLayout host_layout(int B, int H, int H_kv, int S_q, int S_k, int D, const attn_mod_desc* mod,
                       int tpe) {
  HostLayout l;
  const size_t qb = (size_t)B * H * S_q * D * 2, kb = (size_t)B * H_kv * S_k * D * 2;
  size_t at = 0;
  auto take = [&](size_t bytes) {
    const size_t off = at;
    at = align_up(at + bytes, 256);
    return off;
  };
  l.q = take(qb);
  l.k = take(kb);
  l.v = take(kb);
  l.o = take(qb);
  l.lse = take((size_t)B * H * S_q * 4);
  l.doc = take((size_t)B * S_k * 4);
  l.prefix = take((size_t)B * 4);
  l.slopes = take((size_t)H * 4);
  l.blocks_bytes = l.rel_bytes = 0;
  if (mod != nullptr && (mod->mask_flags & ATTN_MASK_BLOCKS))
    l.blocks_bytes = (size_t)(mod->blocks_batched ? B : 1) * ((S_q + kTileM - 1) / kTileM) *
                     ((S_k + kTileN - 1) / kTileN);
  if (mod != nullptr && (mod->score_flags & ATTN_SCORE_RELBIAS))
    l.rel_bytes = (size_t)H * (2 * (size_t)mod->rel_max + 1) * 4;
  l.blocks = take(l.blocks_bytes);
  l.rel = take(l.rel_bytes);
  // one batch entry
  l.mask = take(block_mask_geom(1, S_q, S_k, kernel_mask_flags(mod) & ~kMaskBlocksBatched, tpe).total);
  l.total = at;
  return l;
}

// Grows a slot; its previous call must have finished with the old memory.
attn_status ensure_slot_capacity(HostSlot* sl, size_t bytes) {
  if (sl->bytes >= bytes) return ATTN_OK;
  if (sl->buf != nullptr) {
    if (sl->used && cudaEventSynchronize(sl->done) != cudaSuccess) return ATTN_ERR_CUDA;
    cudaFree(sl->buf);
    sl->buf = nullptr;
    sl->bytes = 0;
  }
  if (cudaMalloc(&sl->buf, bytes) != cudaSuccess) {
    sl->buf = nullptr;
    return ATTN_ERR_CUDA;
  }
  sl->bytes = bytes;
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
      if (value != 0.0 && value != 1.0 && value != 2.0) return ATTN_ERR_INVALID_ARG;
      g_opts.debug_stall = value;
      return ATTN_OK;
    case ATTN_OPT_CTA_PAIR:
      if (value != 0.0 && value != 1.0) return ATTN_ERR_INVALID_ARG;
      g_opts.cta_pair = value;
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
    case ATTN_OPT_CTA_PAIR:
      *value = g_opts.cta_pair;
      return ATTN_OK;
  }
  return ATTN_ERR_INVALID_ARG;
}

size_t attn_block_mask_bytes(int B, int H, int S_q, int S_k, const attn_mod_desc* mod_in) {
  attn_mod_desc mod_buf;
  attn_status lst;
  const attn_mod_desc* mod = load_mod(mod_in, &mod_buf, &lst);
  if (lst != ATTN_OK) return 0;
  if (check_problem(B, H, S_q, S_k, mod) != ATTN_OK) return 0;
  return block_mask_geom(B, S_q, S_k, kernel_mask_flags(mod), mask_tpe(options_snapshot())).total;
}

attn_status attn_build_block_mask(int B, int H, int S_q, int S_k, const attn_mod_desc* mod_in,
                                  void* dst, size_t bytes, attn_stream_t stream) {
  attn_mod_desc mod_buf;
  attn_status lst;
  const attn_mod_desc* mod = load_mod(mod_in, &mod_buf, &lst);
  if (lst != ATTN_OK) return lst;
  attn_status st = check_problem(B, H, S_q, S_k, mod);
  if (st != ATTN_OK) return st;
  if (dst == nullptr || !aligned(dst, 16)) return ATTN_ERR_INVALID_ARG;
  const Options o = options_snapshot();
  const size_t need = block_mask_geom(B, S_q, S_k, kernel_mask_flags(mod), mask_tpe(o)).total;
  if (bytes < need) return ATTN_ERR_INVALID_ARG;
  cudaError_t err = launch_build_block_mask(B, S_q, S_k, mask_params(S_q, S_k, mod),
                                            o.force_partial != 0.0 ? 1 : 0, dst,
                                            reinterpret_cast<cudaStream_t>(stream), mask_tpe(o));
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
  if (h.magic != kBlockMaskMagic || h.version != kBlockMaskVersion || h.total_bytes > bytes ||
      (h.tiles_per_entry != kTilesPerItem && h.tiles_per_entry != kTilesPerQuad))
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
      for (int t = 0; t < h.tiles_per_entry; ++t) {
        if (h.tiles_per_entry * p + t >= h.nQ) continue;
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
                     const attn_mod_desc* mod_in, attn_stream_t stream) {
  attn_mod_desc mod_buf;
  attn_status lst;
  const attn_mod_desc* mod = load_mod(mod_in, &mod_buf, &lst);
  if (lst != ATTN_OK) return lst;
  // ---- host-side validation: nothing is enqueued on failure ------------
  attn_status st = check_problem(B, H, S_q, S_k, mod);
  if (st != ATTN_OK) return st;
  st = check_device_tensors(q, k, v, out, lse, B, H, H_kv, S_q, S_k, D, scale);
  if (st != ATTN_OK) return st;
  const uint32_t mflags = kernel_mask_flags(mod);
  const Options o = options_snapshot();
  const BlockMaskGeom g = block_mask_geom(B, S_q, S_k, mflags, mask_tpe(o));
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
  const void* bmask = (mod != nullptr) ? mod->block_mask : nullptr;
  if (bmask == nullptr) {
    st = ensure_mask_capacity(scr, g.total);
    if (st != ATTN_OK) return st;
  }
  return enqueue_forward(q, k, v, out, lse, B, H, H_kv, S_q, S_k, D, scale, mod, bmask, scr->mask,
                         scr->status, o, s);
}

attn_status attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out, float* lse,
                             int B, int H, int H_kv, int S_q, int S_k, int D, float scale,
                             const attn_mod_desc* mod_in, attn_stream_t stream) {
  attn_mod_desc mod_buf;
  attn_status lst;
  const attn_mod_desc* mod = load_mod(mod_in, &mod_buf, &lst);
  if (lst != ATTN_OK) return lst;
  // ---- host-side validation (same rules as attn_fwd) -----------------------
  attn_status st = check_problem(B, H, S_q, S_k, mod);
  if (st != ATTN_OK) return st;
  st = check_device_tensors(q, k, v, out, lse, B, H, H_kv, S_q, S_k, D, scale);
  if (st != ATTN_OK) return st;
  // The block mask is always built into the fixed scratch array.
  if (mod != nullptr && mod->block_mask != nullptr) return ATTN_ERR_INVALID_ARG;
  const uint32_t mflags = kernel_mask_flags(mod);
  const Options o = options_snapshot();
  const BlockMaskGeom g = block_mask_geom(B, S_q, S_k, mflags, mask_tpe(o));
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
  return enqueue_forward(q, k, v, out, lse, B, H, H_kv, S_q, S_k, D, scale, mod, nullptr, bmask,
                         status, o, s);
}

attn_status attn_get_noalloc_status(attn_stream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  void* scratch = nullptr;
  attn_status st = noalloc_scratch(dev, &scratch);
  if (st != ATTN_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  DeviceStatus h;
  if (cudaMemcpy(&h, scratch, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (h.code != 0 && cudaMemset(scratch, 0, sizeof(DeviceStatus)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return static_cast<attn_status>(h.code);
}

attn_status attn_fwd_host(const void* q, const void* k, const void* v, void* out, float* lse,
                          int B, int H, int H_kv, int S_q, int S_k, int D, float scale,
                          const attn_mod_desc* mod_in, attn_stream_t stream) {
  attn_mod_desc mod_buf;
  attn_status lst;
  const attn_mod_desc* mod = load_mod(mod_in, &mod_buf, &lst);
  if (lst != ATTN_OK) return lst;
  // ---- host-side validation: nothing is enqueued on failure --------------
  attn_status st = check_problem(B, H, S_q, S_k, mod);
  if (st != ATTN_OK) return st;
  st = check_tensors(q, k, v, out, lse, B, H, H_kv, S_q, S_k, D, scale);
  if (st != ATTN_OK) return st;
  if (mod != nullptr && mod->block_mask != nullptr) return ATTN_ERR_INVALID_ARG;
  const Options o = options_snapshot();
  const HostLayout lay = host_layout(B, H, H_kv, S_q, S_k, D, mod, mask_tpe(o));

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  DeviceScratch* scr = nullptr;
  st = scratch_for(dev, &scr);
  if (st != ATTN_OK) return st;
  HostPipe* pipe = nullptr;
  st = host_pipe(dev, &pipe);
  if (st != ATTN_OK) return st;
  std::lock_guard<std::mutex> lk(pipe->mu);
  HostSlot& slot = pipe->slot[pipe->next];
  st = ensure_slot_capacity(&slot, lay.total);
  if (st != ATTN_OK) return st;
  pipe->next ^= 1;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(slot.buf);
  auto ck = [](cudaError_t e) { return e == cudaSuccess; };
  const uint32_t mflags = kernel_mask_flags(mod);
  const uint32_t sflags = mod ? mod->score_flags : 0u;
  const int group = H / H_kv;
  const size_t q_head = (size_t)S_q * D * 2, k_head = (size_t)S_k * D * 2;
  const size_t l_head = (size_t)S_q * 4;
  // Inputs start after the caller's earlier work on `stream` and after this
  // slot's previous call has copied its results out.
  bool ok = ck(cudaEventRecord(pipe->user, s)) && ck(cudaStreamWaitEvent(pipe->h2d, pipe->user, 0));
  if (ok && slot.used) ok = ck(cudaStreamWaitEvent(pipe->h2d, slot.done, 0));
  if (ok && (mflags & ATTN_MASK_DOCUMENT))
    ok = ck(cudaMemcpyAsync(base + lay.doc, mod->doc_ids, (size_t)B * S_k * 4,
                            cudaMemcpyHostToDevice, pipe->h2d));
  if (ok && (mflags & ATTN_MASK_PREFIX_LM))
    ok = ck(cudaMemcpyAsync(base + lay.prefix, mod->prefix_len, (size_t)B * 4,
                            cudaMemcpyHostToDevice, pipe->h2d));
  const bool alibi = (sflags & ATTN_SCORE_ALIBI) != 0;
  if (ok && alibi && mod->alibi_slopes != nullptr)
    ok = ck(cudaMemcpyAsync(base + lay.slopes, mod->alibi_slopes, (size_t)H * 4,
                            cudaMemcpyHostToDevice, pipe->h2d));
  if (ok && lay.blocks_bytes)
    ok = ck(cudaMemcpyAsync(base + lay.blocks, mod->blocks, lay.blocks_bytes,
                            cudaMemcpyHostToDevice, pipe->h2d));
  if (ok && lay.rel_bytes)
    ok = ck(cudaMemcpyAsync(base + lay.rel, mod->rel_bias, lay.rel_bytes, cudaMemcpyHostToDevice,
                            pipe->h2d));
  if (!ok) return ATTN_ERR_CUDA;
  // Slices of heads run as separate forwards, so the default ALiBi slopes
  // (which depend on the head's index among all H) are written out once.
  float* dslopes = reinterpret_cast<float*>(base + lay.slopes);
  if (alibi && mod->alibi_slopes == nullptr &&
      launch_default_alibi_slopes(dslopes, H, pipe->comp) != cudaSuccess)
    return ATTN_ERR_CUDA;

  // The call runs in chunks -- one batch entry and a run of K/V heads with
  // their query heads each -- so chunk c's compute overlaps chunk c+1's input
  // copy and chunk c-1's output copy.  The host link, not the tensor cores,
  // bounds this path; about eight chunks hide nearly all of the compute.
  const int units = B * H_kv;
  const int per = (units + kHostChunks - 1) / kHostChunks;  // K/V heads per chunk
  const bool per_batch = mask_per_batch(mflags);
  const size_t map_bytes = (size_t)((S_q + kTileM - 1) / kTileM) * ((S_k + kTileN - 1) / kTileN);
  int mask_b = -1;  // batch entry whose block mask is in the slot
  for (int b = 0; b < B && ok; ++b) {
    for (int kv0 = 0; kv0 < H_kv && ok; kv0 += per) {
      const int kv1 = kv0 + per < H_kv ? kv0 + per : H_kv;
      const int nkv = kv1 - kv0, nh = nkv * group;
      const size_t qh0 = (size_t)b * H + (size_t)kv0 * group;  // first query head (flat)
      const size_t kh0 = (size_t)b * H_kv + (size_t)kv0;       // first K/V head (flat)
      ok = ck(cudaMemcpyAsync(base + lay.q + qh0 * q_head, static_cast<const char*>(q) + qh0 * q_head,
                              (size_t)nh * q_head, cudaMemcpyHostToDevice, pipe->h2d)) &&
           ck(cudaMemcpyAsync(base + lay.k + kh0 * k_head, static_cast<const char*>(k) + kh0 * k_head,
                              (size_t)nkv * k_head, cudaMemcpyHostToDevice, pipe->h2d)) &&
           ck(cudaMemcpyAsync(base + lay.v + kh0 * k_head, static_cast<const char*>(v) + kh0 * k_head,
                              (size_t)nkv * k_head, cudaMemcpyHostToDevice, pipe->h2d)) &&
           ck(cudaEventRecord(pipe->in, pipe->h2d)) &&
           ck(cudaStreamWaitEvent(pipe->comp, pipe->in, 0));
      if (!ok) break;
      // this chunk as a problem of its own: batch 1, its heads, batch b's
      // mask arrays
      attn_mod_desc cm;
      memset(&cm, 0, sizeof(cm));
      if (mod != nullptr) cm = *mod;
      cm.version = ATTN_MOD_DESC_VERSION;
      cm.block_mask = nullptr;
      cm.block_mask_bytes = 0;
      if (mflags & ATTN_MASK_DOCUMENT)
        cm.doc_ids = reinterpret_cast<const int32_t*>(base + lay.doc) + (size_t)b * S_k;
      if (mflags & ATTN_MASK_PREFIX_LM)
        cm.prefix_len = reinterpret_cast<const int32_t*>(base + lay.prefix) + b;
      if (alibi) cm.alibi_slopes = dslopes + (size_t)kv0 * group;
      if (mflags & ATTN_MASK_BLOCKS) {  // batch b's map (one batch entry here)
        cm.blocks = reinterpret_cast<const uint8_t*>(base + lay.blocks) +
                    (mod->blocks_batched ? (size_t)b * map_bytes : 0);
        cm.blocks_batched = 0;
      }
      if (sflags & ATTN_SCORE_RELBIAS)
        cm.rel_bias = reinterpret_cast<const float*>(base + lay.rel) +
                      (size_t)kv0 * group * (2 * (size_t)mod->rel_max + 1);
      // one block mask per batch entry (or one for all when the mask does
      // not depend on the batch); the stream orders each rebuild after the
      // forwards that read the previous one
      const int want_b = per_batch ? b : 0;
      if (mask_b != want_b) {
        if (launch_build_block_mask(1, S_q, S_k, mask_params(S_q, S_k, &cm),
                                    o.force_partial != 0.0 ? 1 : 0, base + lay.mask, pipe->comp,
                                    mask_tpe(o)) != cudaSuccess)
          return ATTN_ERR_CUDA;
        mask_b = want_b;
      }
      float* dl = lse != nullptr ? reinterpret_cast<float*>(base + lay.lse) + qh0 * S_q : nullptr;
      st = enqueue_forward(base + lay.q + qh0 * q_head, base + lay.k + kh0 * k_head,
                           base + lay.v + kh0 * k_head, base + lay.o + qh0 * q_head, dl, 1, nh,
                           nkv, S_q, S_k, D, scale, &cm, base + lay.mask, nullptr, scr->status, o,
                           pipe->comp);
      if (st != ATTN_OK) return st;
      ok = ck(cudaEventRecord(pipe->comp_ev, pipe->comp)) &&
           ck(cudaStreamWaitEvent(pipe->d2h, pipe->comp_ev, 0)) &&
           ck(cudaMemcpyAsync(static_cast<char*>(out) + qh0 * q_head, base + lay.o + qh0 * q_head,
                              (size_t)nh * q_head, cudaMemcpyDeviceToHost, pipe->d2h));
      if (ok && lse != nullptr)
        ok = ck(cudaMemcpyAsync(lse + qh0 * S_q, dl, (size_t)nh * l_head, cudaMemcpyDeviceToHost,
                                pipe->d2h));
    }
  }
  // `stream` continues once every result is in host memory
  if (ok) ok = ck(cudaEventRecord(slot.done, pipe->d2h));
  if (ok) slot.used = true;
  if (ok) ok = ck(cudaStreamWaitEvent(s, slot.done, 0));
  return ok ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* out,
                     const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                     int H, int H_kv, int S_q, int S_k, int D, float scale,
                     const attn_mod_desc* mod_in, attn_stream_t stream) {
  attn_mod_desc mod_buf;
  attn_status lst;
  const attn_mod_desc* mod = load_mod(mod_in, &mod_buf, &lst);
  if (lst != ATTN_OK) return lst;
  // ---- host-side validation: nothing is enqueued on failure --------------
  attn_status st = check_problem(B, H, S_q, S_k, mod);
  if (st != ATTN_OK) return st;
  st = check_device_tensors(q, k, v, out, lse, B, H, H_kv, S_q, S_k, D, scale);
  if (st != ATTN_OK) return st;
  if (lse == nullptr || dout == nullptr || dq == nullptr || dk == nullptr || dv == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if (!aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16))
    return ATTN_ERR_INVALID_ARG;
  if (mod != nullptr && mod->block_mask != nullptr) return ATTN_ERR_INVALID_ARG;
  const size_t qb = (size_t)B * H * S_q * D * 2, kb = (size_t)B * H_kv * S_k * D * 2;
  const size_t lb = (size_t)B * H * S_q * 4;
  const void* ins[6] = {q, k, v, out, lse, dout};
  const size_t in_b[6] = {qb, kb, kb, qb, lb, qb};
  void* outs[3] = {dq, dk, dv};
  const size_t out_b[3] = {qb, kb, kb};
  for (int o = 0; o < 3; ++o) {
    for (int i = 0; i < 6; ++i)
      if (overlaps(outs[o], out_b[o], ins[i], in_b[i])) return ATTN_ERR_INVALID_ARG;
    for (int o2 = 0; o2 < o; ++o2)
      if (overlaps(outs[o], out_b[o], outs[o2], out_b[o2])) return ATTN_ERR_INVALID_ARG;
  }

  // ---- device work -------------------------------------------------------
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  DeviceScratch* scr = nullptr;
  st = scratch_for(dev, &scr);
  if (st != ATTN_OK) return st;
  const uint32_t mflags = kernel_mask_flags(mod);
  const BlockMaskGeom g = block_mask_geom(B, S_q, S_k, mflags);
  const BlockMaskTGeom gt = block_mask_t_geom(B, S_q, S_k, mflags);
  const size_t off_t = align_up(g.total, 256);
  const size_t off_r = align_up(off_t + gt.total, 256);
  const size_t total = off_r + bwd_rowstat_bytes(B, H, S_q);
  void* buf = nullptr;
  st = bwd_scratch(dev, total, &buf);
  if (st != ATTN_OK) return st;
  char* base = static_cast<char*>(buf);
  const Options o = options_snapshot();
  const MaskParams mp = mask_params(S_q, S_k, mod);
  const int fp = o.force_partial != 0.0 ? 1 : 0;
  if (launch_build_block_mask(B, S_q, S_k, mp, fp, base, s) != cudaSuccess ||
      launch_build_block_mask_t(B, S_q, S_k, mp, fp, base, base + off_t, s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  BwdArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.dout = dout;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
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
  if (mod && (mod->score_flags & ATTN_SCORE_RELBIAS)) {
    a.rel_bias = mod->rel_bias;
    a.rel_max = mod->rel_max;
  }
  a.block_mask = base;
  a.block_mask_t = base + off_t;
  a.rowstat = reinterpret_cast<float*>(base + off_r);
  a.status = scr->status;
  a.wait_budget_ms = o.wait_budget_ms;
  a.force_partial = fp;
  a.debug_stall = (o.debug_stall == 1.0 || o.debug_stall == 2.0) ? (int)o.debug_stall : 0;
  return launch_attn_bwd(a, s) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // extern "C"
