// attn_bwd_sm103.cu -- attention backward for GB300 (sm_103a): dQ, dK, dV.
//
// The gradients of the forward (softmax attention with the same masks and
// score mods), by the chain rule:
//   P  = exp(S' - LSE)            S' the modified score, LSE from the forward
//   dP = dO V^T
//   dS = P * (dP - rowsum(dO * O)) * dS'/dS
//   dQ = scale * dS K,   dK = scale * dS^T Q,   dV = P^T dO
// ("FlashAttention-4 explained", section "FlashAttention-4: Built for
// Blackwell", names the backward as the step after the forward; the
// recomputation of P from the saved LSE instead of storing it is the same
// principle as "Enter Tri Dao and FlashAttention": the score matrix never
// goes to HBM.)
//
// Three kernels:
//   bwd_prep_kernel   per query row: -LSE in log2 units and -(dO . O),
//                     padded to whole 128-row tiles (padding rows get
//                     -inf / 0, so they contribute P = 0 without a mask);
//                     negated so that the elementwise steps are additions
//                     (paired fp32 instructions)
//   bwd_dq_kernel     one 128-row query tile per work item: for each key tile
//                     of its block-mask list, S = Q K^T and dP = dO V^T into
//                     Tensor Memory, dS by the elementwise warpgroup (one
//                     thread per query row), dQ += dS K accumulated in Tensor
//                     Memory
//   bwd_dkdv_kernel   one 128-key tile per work item (K/V head, all query
//                     heads of its group): S^T = K Q^T and dP^T = V dO^T, then
//                     P^T and dS^T by the elementwise warpgroup (one thread
//                     per key), dV += P^T dO and dK += dS^T Q accumulated in
//                     Tensor Memory (GQA sums over the group in place)
// Neither kernel uses atomics: every output row is written once by the work
// item that owns it, so results are deterministic.
//
// Warp roles (320 threads): warps 0-7 elementwise in two warpgroups, warp 8
// TMA loads, warp 9 allocates Tensor Memory and issues the MMAs (168
// registers a thread: moving registers from a third warpgroup to the
// elementwise ones with setmaxnreg removed the last spills of the dK/dV
// kernel but measured 3-4% slower).  Warps w
// and w + 4 share Tensor Memory lane quarter w & 3 (32 rows of the tile) and
// split its 128 columns: warpgroup 0 takes columns [0, 64), warpgroup 1
// [64, 128).  No elementwise step reduces along a row (P = exp(S - LSE) with
// LSE known, dS = P (dP - Delta) with Delta known), so the halves are
// independent, and two warps per SM sub-partition hide each other's latency.
// Each half packs its bf16 results (P^T, dS, dS^T) over its own columns,
// half 0 at packed columns [32, 64) and half 1 at [64, 96), so the packed
// 128-wide operand is contiguous at column 32 for the MMA that reads it.
// Every wait is bounded like the forward's: on expiry the kernel records
// ATTN_ERR_TIMEOUT and returns.
#include <atomic>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <float.h>
#include <math.h>

#include "attn_internal.h"
#include "sm103_ptx.cuh"
#include "tanh_poly.h"

namespace attn {

namespace {

constexpr int kBThreads = 320;
constexpr int kBLoadWarp = 8;
constexpr int kBMmaWarp = 9;

constexpr int kBCols = 64;      // columns of a tile per elementwise half
constexpr uint32_t kBPack = 32;  // packed operand: Tensor Memory columns [32, 96)
constexpr uint32_t kBTmemCols = 512;
constexpr float kBLog2e = 1.4426950408889634f;

enum BSite : int {
  kBSiteHeader = 101,
  kBSiteLoad = 110,
  kBSiteMma = 120,
  kBSiteElem = 130,
  kBSiteDrain = 140,
  kBSiteDebugStall = 150,  // + 1 in the dQ kernel, + 2 in the dK/dV kernel
};

template <int D>
struct BCfg {
  static constexpr int kHalfBytes = kTileM * 64 * 2;  // 128 rows x 64 bf16, 128-byte swizzle
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = kHalves * kHalfBytes;
  // bwd_dq_kernel: Q, dO, a ring of K tiles, a ring of V tiles (K is read
  // by S and dQ, V only by dP, so V tiles are released earlier and need
  // fewer stages)
  static constexpr int kDqQ = 0;
  static constexpr int kDqDo = kTileBytes;
  static constexpr int kDqKStages = 3;
  static constexpr int kDqVStages = 2;
  static constexpr int kDqK = 2 * kTileBytes;
  static constexpr int kDqV = kDqK + kDqKStages * kTileBytes;
  static constexpr int kDqBar = kDqV + kDqVStages * kTileBytes;
  // bwd_dkdv_kernel: K, V, then two stages of (Q, dO, LSE2[128], Delta[128])
  static constexpr int kKvK = 0;
  static constexpr int kKvV = kTileBytes;
  static constexpr int kKvStage0 = 2 * kTileBytes;
  static constexpr int kKvStageBytes = 2 * kTileBytes + 1024;
  static constexpr int kKvBar = kKvStage0 + 2 * kKvStageBytes;
  static constexpr int kNumBars = 24;
  static constexpr int kSmemDq = kDqBar + 8 * kNumBars + 16;
  static constexpr int kSmemKv = kKvBar + 8 * kNumBars + 16;
  static constexpr int kSmemAllocDq = kSmemDq + 1024;
  static constexpr int kSmemAllocKv = kSmemKv + 1024;
};

struct BParams {
  CUtensorMap tmap_q;
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  CUtensorMap tmap_do;
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const float* nlse2;   // [B*H][nQ*128] -LSE * log2(e)
  const float* ndelta;  // [B*H][nQ*128] -(dO . O)
  int B, H, H_kv, S_q, S_k, group, nQ, nK, nP, bm;
  float scale, scale_log2, softcap;
  uint32_t mask_flags;
  int window, q_offset;
  const int32_t* doc_ids;
  const int32_t* prefix_len;
  const int32_t* doc_lo;
  const int32_t* doc_hi;
  const float* alibi_slopes;
  int alibi_on;           // the ALiBi variant also serves a bias table alone
  const float* rel_bias;  // [H][2 rel_max + 1], or null
  int rel_max;
  const BlockMaskHeader* hdr;
  const int32_t* cnt;      // forward block mask: per query-tile pair
  const uint32_t* list;
  const int32_t* cnt_t;    // transposed: per key tile
  const uint32_t* list_t;
  int n_items;
  DeviceStatus* status;
  uint64_t budget_ns;
  int debug_stall;  // test hook: 1 = the dQ kernel, 2 = the dK/dV kernel
  // soft cap on the FMA pipes, as in the forward: t = y Q(y^2) for the
  // score y in the units 2 log2(e) x / cap while |y| <= tlim
  float tq[3];
  float tlim;
};

struct BCtl {
  volatile int* abort;
  uint32_t abort_smem;
  DeviceStatus* status;
  uint64_t budget_ns;
};

__device__ __noinline__ void breport(const BCtl& c, int code, int site, int detail) {
  if (atomicCAS(&c.status->code, 0, code) == 0) {
    c.status->where = site;
    c.status->block = blockIdx.x;
    c.status->detail = detail;
  }
  *c.abort = 1;
}

// Bounded mbarrier wait (see the forward kernel's): false on timeout or when
// another role has aborted.
__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, const BCtl& c, int site) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = 0;
  for (uint32_t spin = 1;; ++spin) {
    if (ptx::mbar_try_wait_hint(bar, parity, 20000)) return true;
    if ((spin & 15) == 0) {
      if (ptx::ld_volatile_shared(c.abort_smem)) return false;
      const uint64_t now = ptx::globaltimer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > c.budget_ns) {
        breport(c, ATTN_ERR_TIMEOUT, site, (int)parity);
        return false;
      }
    }
  }
}

template <int D>
struct BDesc {
  static constexpr uint64_t kKMajor = ptx::smem_desc_sw128(0, 16, 1024);
  static constexpr uint64_t kMNMajor = ptx::smem_desc_sw128(0, BCfg<D>::kHalfBytes, 1024);
};

// C = A B^T over the head dimension with both operands K-major 128 x D
// tiles in shared memory (8 or 4 MMAs, K = 16 each).  Warp-wide.
template <int D>
__device__ __forceinline__ void mma_nt(uint32_t tmem_c, uint64_t a_desc, uint64_t b_desc) {
  constexpr uint32_t idesc = ptx::idesc_bf16_f32(kTileM, kTileN, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = (uint64_t)(((kk / 4) * BCfg<D>::kHalfBytes + (kk % 4) * 32) >> 4);
    ptx::mma_ss_elect(tmem_c, a_desc + off, b_desc + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// C (+)= A B with A 128 x 128 bf16 packed in Tensor Memory (the 64 packed
// columns at tmem_a) and B a 128 x D tile in shared memory read MN-major.
template <int D>
__device__ __forceinline__ void mma_tn(uint32_t tmem_c, uint32_t tmem_a, uint64_t b_desc,
                                       bool accumulate) {
  constexpr uint32_t idesc = ptx::idesc_bf16_f32(kTileM, D, true);
#pragma unroll
  for (int kk = 0; kk < kTileN / 16; ++kk)
    ptx::mma_ts_elect(tmem_c, tmem_a + (uint32_t)(kk * 8), b_desc + (uint64_t)((kk * 2048) >> 4),
                      idesc, (accumulate || kk > 0) ? 1u : 0u);
}

// 32 bf16 values (16 packed words) to a row: whole 32-byte sectors when the
// tensor is 32-byte aligned (rows are), 16-byte stores otherwise.
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const uint32_t (&pk)[16],
                                            bool al32) {
  if (al32) {
    ptx::stg_v8(dst, pk);
    ptx::stg_v8(dst + 16, pk + 8);
  } else {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int c = 0; c < 4; ++c)
      d4[c] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
  }
}

// After an abort, let a loader's copies in flight land before the CTA
// exits: wait (bounded) for the last phase issued on each of n_stages
// barriers that saw `issued` loads in total (round-robin).
__device__ __forceinline__ void drain_loads(uint32_t bar0, int n_stages, uint32_t issued,
                                            uint64_t budget_ns) {
  const uint32_t first = issued > (uint32_t)n_stages ? issued - n_stages : 0;
  for (uint32_t c = first; c < issued; ++c) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar0 + 8u * (c % n_stages), (c / n_stages) & 1) &&
           ptx::globaltimer_ns() - t0 < budget_ns) {
    }
  }
}

// Static snake schedule over the items (as the forward's).
__device__ __forceinline__ int bitem_of(int r) {
  const int G = gridDim.x, c = blockIdx.x;
  return r * G + ((r & 1) ? (G - 1 - c) : c);
}

// The score transform in log2 units, as in the forward kernel.
struct ScoreMod {
  float sc, slope2, capl2, inv_capl2;
};
template <bool ALIBI, bool SOFTCAP>
__device__ __forceinline__ float score_t(float s, float bias_pos, const ScoreMod& m) {
  float x = s * m.sc;
  if constexpr (ALIBI) x = fmaf(m.slope2, bias_pos, x);
  if constexpr (SOFTCAP) {
    const float e = ptx::ex2_approx(x);
    x = m.capl2 * (1.0f - 2.0f * ptx::rcp_approx(e + 1.0f));
  }
  return x;
}
// The score transform of N columns in place, their bias positions
// pos0 + step * c: as score_t, except that a soft cap whose scores all lie
// within the polynomial's range for every lane of the warp (always, for
// scores of ordinary size) is evaluated as t = y Q(y^2) on the FMA pipes
// (tanh_poly.h; paired fp32 instructions) instead of from the exp2 and
// reciprocal units, whose reciprocal runs at half the exp2 rate.
template <bool ALIBI, bool SOFTCAP, int N>
__device__ __forceinline__ void score_cols(float (&tv)[N], float pos0, float step,
                                           const ScoreMod& m, const BParams& p) {
  if constexpr (!SOFTCAP) {
#pragma unroll
    for (int c = 0; c < N; ++c) tv[c] = score_t<ALIBI, SOFTCAP>(tv[c], pos0 + step * (float)c, m);
  } else {
    float mx = -INFINITY, mn = INFINITY;
#pragma unroll
    for (int c = 0; c < N; ++c) {
      float y = tv[c] * m.sc;
      if constexpr (ALIBI) y = fmaf(m.slope2, pos0 + step * (float)c, y);
      tv[c] = y;
      mx = fmaxf(mx, y);
      mn = fminf(mn, y);
    }
    if (__all_sync(0xffffffffu, mx <= p.tlim && mn >= -p.tlim)) {
      const uint64_t q2 = ptx::f2(p.tq[2], p.tq[2]), q1 = ptx::f2(p.tq[1], p.tq[1]),
                     q0 = ptx::f2(p.tq[0], p.tq[0]);
#pragma unroll
      for (int c = 0; c < N; c += 2) {
        const uint64_t y2 = ptx::f2(tv[c], tv[c + 1]);
        const uint64_t w2 = ptx::fmul2(y2, y2);
        uint64_t r2 = ptx::ffma2(w2, q2, q1);
        r2 = ptx::ffma2(r2, w2, q0);
        ptx::f2_split(ptx::fmul2(y2, r2), tv[c], tv[c + 1]);
      }
    } else {
#pragma unroll
      for (int c = 0; c < N; ++c) {
        const float e = ptx::ex2_approx(tv[c]);
        tv[c] = m.capl2 * (1.0f - 2.0f * ptx::rcp_approx(e + 1.0f));
      }
    }
  }
}

template <bool ALIBI, bool SOFTCAP>
__device__ __forceinline__ ScoreMod make_mod(const BParams& p, int h) {
  ScoreMod m;
  m.sc = SOFTCAP ? p.scale * (2.0f * kBLog2e / p.softcap) : p.scale_log2;
  m.capl2 = p.softcap * kBLog2e;
  m.inv_capl2 = SOFTCAP ? 1.0f / m.capl2 : 0.f;
  m.slope2 = 0.f;
  if constexpr (ALIBI) {
    if (p.alibi_on) {
      const float mh =
          p.alibi_slopes ? p.alibi_slopes[h] : exp2f(-8.0f * (float)(h + 1) / (float)p.H);
      m.slope2 = SOFTCAP ? mh * (2.0f * kBLog2e / p.softcap) : mh * kBLog2e;
    }
  }
  return m;
}

// Adds the relative-position bias of head h to raw scores tv[0..N-1] whose
// relative positions (kpos - qpos) are pos0 + step * c, pre-divided by the
// score scale so that score_t applies it as table * (units of t); a
// uniform branch around its own loop keeps the other loops branch-free.
template <bool ALIBI, bool SOFTCAP, int N>
__device__ __forceinline__ void add_rel_bias(float (&tv)[N], const BParams& p, int h, int pos0,
                                             int step, const ScoreMod& m) {
  if constexpr (ALIBI) {
    if (p.rel_bias == nullptr) return;
    const float* row = p.rel_bias + (size_t)h * (2 * (size_t)p.rel_max + 1);
    const float rs = (SOFTCAP ? 2.0f * kBLog2e / p.softcap : kBLog2e) / m.sc;
    // beyond +-R of every position of the warp the clamped bias is one entry
    const int lo_r = min(pos0, pos0 + step * (N - 1)), hi_r = max(pos0, pos0 + step * (N - 1));
    float cst = 0.f;
    bool flat = true;
    if (__all_sync(0xffffffffu, hi_r <= -p.rel_max)) {
      cst = __ldg(row);
    } else if (__all_sync(0xffffffffu, lo_r >= p.rel_max)) {
      cst = __ldg(row + 2 * p.rel_max);
    } else {
      flat = false;
    }
    if (flat) {
      const float add = cst * rs;
#pragma unroll
      for (int c = 0; c < N; ++c) tv[c] += add;
      return;
    }
#pragma unroll
    for (int c = 0; c < N; ++c) {
      const int r = min(max(pos0 + step * c, -p.rel_max), p.rel_max);
      tv[c] = fmaf(__ldg(row + r + p.rel_max), rs, tv[c]);
    }
  }
}

// Visible key interval of query row i (forward orientation).
__device__ __forceinline__ void row_keys(const BParams& p, int b, int i, bool docs_sorted,
                                         int& lo, int& hi) {
  const int qpos = i + p.q_offset;
  lo = 0;
  hi = p.S_k - 1;
  if (p.mask_flags & ATTN_MASK_CAUSAL) hi = min(hi, qpos);
  if (p.mask_flags & ATTN_MASK_WINDOW) {
    lo = max(lo, qpos - p.window + 1);
    hi = min(hi, qpos);
  }
  if (p.mask_flags & ATTN_MASK_PREFIX_LM) hi = min(hi, max(qpos, p.prefix_len[b] - 1));
  if ((p.mask_flags & ATTN_MASK_DOCUMENT) && docs_sorted && i < p.S_q) {
    const size_t di = (size_t)b * p.S_k + (size_t)i;
    lo = max(lo, p.doc_lo[di]);
    hi = min(hi, p.doc_hi[di]);
  }
}

// Query rows that see key j (transposed orientation): the interval
// [ilo, ihi] of query indices, from the same mask rules.
__device__ __forceinline__ void key_rows(const BParams& p, int b, int j, bool docs_sorted,
                                         int& ilo, int& ihi) {
  long long lo = 0, hi = (long long)p.S_q - 1;
  const long long first = (long long)j - p.q_offset;  // query index whose qpos == j
  if (p.mask_flags & ATTN_MASK_CAUSAL) lo = max(lo, first);
  if (p.mask_flags & ATTN_MASK_WINDOW) {
    lo = max(lo, first);
    hi = min(hi, first + p.window - 1);
  }
  if ((p.mask_flags & ATTN_MASK_PREFIX_LM) && !(j < p.prefix_len[b])) lo = max(lo, first);
  if ((p.mask_flags & ATTN_MASK_DOCUMENT) && docs_sorted && j < p.S_k) {
    const size_t di = (size_t)b * p.S_k + (size_t)j;
    lo = max(lo, (long long)p.doc_lo[di]);
    hi = min(hi, (long long)p.doc_hi[di]);
  }
  ilo = (int)max(lo, -1ll);
  ihi = (int)min(hi, (long long)p.S_q);
}

// ---------------------------------------------------------------- prep ----
// nlse2[r] = -LSE * log2(e) (-inf where the row has no visible key or r is
// padding); ndelta[r] = -(dO_r . O_r) (0 for padding).  Four threads per row,
// each with D/4 elements of O and of dO in flight as 16-byte loads (the
// kernel only streams O and dO once, so it is bound by HBM).
constexpr int kPrepTpr = 4;                     // threads per row
constexpr int kPrepRows = 256 / kPrepTpr;       // rows per 256-thread block
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* out,
                                                       const __nv_bfloat16* dout,
                                                       const float* lse, float* nlse2,
                                                       float* ndelta, int BH, int S_q, int nQ) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  constexpr int kVec = D / (8 * kPrepTpr);  // 16-byte vectors per thread and tensor
  const long long per = (long long)nQ * kTileM;
  const long long rows = (long long)BH * per;
  const long long r = (long long)blockIdx.x * kPrepRows + (threadIdx.x / kPrepTpr);
  const int q = threadIdx.x % kPrepTpr;
  const bool in = r < rows;
  const long long bh = in ? r / per : 0;
  const int i = in ? (int)(r % per) : S_q;
  float acc = 0.f;
  if (i < S_q) {
    const size_t base = ((size_t)bh * S_q + (size_t)i) * D + (size_t)q * (D / kPrepTpr);
    const uint4* o4 = reinterpret_cast<const uint4*>(out + base);
    const uint4* g4 = reinterpret_cast<const uint4*>(dout + base);
    uint4 ov[kVec], gv[kVec];
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      ov[v] = __ldg(o4 + v);
      gv[v] = __ldg(g4 + v);
    }
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      const __nv_bfloat162* a = reinterpret_cast<const __nv_bfloat162*>(&ov[v]);
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&gv[v]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __bfloat1622float2(a[e]), fb = __bfloat1622float2(b[e]);
        acc = fmaf(fa.x, fb.x, acc);
        acc = fmaf(fa.y, fb.y, acc);
      }
    }
  }
  // the row's four partial sums (lanes 4k .. 4k+3 of the warp)
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  if (in && q == 0) {
    float nl2 = -INFINITY;
    if (i < S_q) {
      const float l = lse[(size_t)bh * S_q + (size_t)i];
      if (l != -INFINITY) nl2 = -(l * kBLog2e);
    }
    nlse2[r] = nl2;
    ndelta[r] = -acc;
  }
}

// ------------------------------------------------------------------ dQ ----
template <int D, bool ALIBI, bool SOFTCAP>
__global__ void __launch_bounds__(kBThreads, 1) bwd_dq_kernel(const __grid_constant__ BParams p) {
  using C = BCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  ptx::griddep_wait();
  const int docs_sorted = p.hdr->docs_sorted;

  auto bar = [&](int i) { return sbase + (uint32_t)(C::kDqBar + 8 * i); };
  constexpr int KS = C::kDqKStages, VS = C::kDqVStages;
  // KF/KE: K ring (KS each), VF/VE: V ring (VS each), DPF: one per dP buffer
  enum { QF = 0, QE = 1, SF = 2, DSF = 3, DQF = 4, DQE = 5, DRAIN = 6, SCON = 7, DPF = 8,
         KF = 10, KE = KF + KS, VF = KE + KS, VE = VF + VS, NEVER = VE + VS };
  static_assert(NEVER < C::kNumBars, "barrier slots");
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::kDqBar + 8 * C::kNumBars);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::kDqBar + 8 * C::kNumBars + 4);
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(QF), 1);
    ptx::mbar_init(bar(QE), 1);
    for (int s = 0; s < KS; ++s) {
      ptx::mbar_init(bar(KF + s), 1);
      ptx::mbar_init(bar(KE + s), 1);
    }
    for (int s = 0; s < VS; ++s) {
      ptx::mbar_init(bar(VF + s), 1);
      ptx::mbar_init(bar(VE + s), 1);
    }
    // one arrival per elementwise warp
    ptx::mbar_init(bar(SF), 1);
    ptx::mbar_init(bar(DSF), 8);
    ptx::mbar_init(bar(DQF), 1);
    ptx::mbar_init(bar(DQE), 8);
    ptx::mbar_init(bar(DPF), 1);
    ptx::mbar_init(bar(DPF + 1), 1);
    ptx::mbar_init(bar(SCON), 8);
    ptx::mbar_init(bar(DRAIN), 1);
    ptx::mbar_init(bar(NEVER), 1);  // the test hook's: nothing arrives on it
    *s_abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kBMmaWarp) {
    ptx::tmem_alloc(ptx::smem_addr(s_tmem), kBTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const BCtl ctl{s_abort, sbase + (uint32_t)(C::kDqBar + 8 * C::kNumBars + 4), p.status,
                 p.budget_ns};

  // Item w -> (b, h, query tile); its key tiles are the forward mask's list
  // of the tile's pair, skipping the entries EMPTY for this tile.
  struct It {
    int b, h, qt, t, n;
    const uint32_t* lst;
  };
  auto item = [&](int w) {
    It it;
    it.qt = w % p.nQ;
    const int bh = w / p.nQ;
    it.b = bh / p.H;
    it.h = bh % p.H;
    it.t = it.qt & 1;
    const int e = (p.bm == 1 ? 0 : it.b) * p.nP + (it.qt >> 1);
    it.n = p.cnt[e];
    it.lst = p.list + (size_t)e * p.nK;
    return it;
  };
  auto nonempty = [&](const It& it) {
    int m = 0;
    for (int j = 0; j < it.n; ++j) m += entry_cls(it.lst[j], it.t) != kEmpty;
    return m;
  };

  if (warp >= 8) {
  if (warp == kBLoadWarp) {
    if (lane == 0) {
      ptx::prefetch_tmap(&p.tmap_q);
      ptx::prefetch_tmap(&p.tmap_do);
      ptx::prefetch_tmap(&p.tmap_k);
      ptx::prefetch_tmap(&p.tmap_v);
      const uint64_t pol = ptx::policy_evict_last();
      uint32_t kv_cnt = 0, q_issued = 0, v_issued = 0;
      int act = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int w = bitem_of(r);
        if (w >= p.n_items) break;
        const It it = item(w);
        if (nonempty(it) == 0) continue;
        if (act > 0) ok = bwait(bar(QE), (act - 1) & 1, ctl, kBSiteLoad);
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(bar(QF), 2 * C::kTileBytes);
        q_issued = act + 1;
        for (int hx = 0; hx < C::kHalves; ++hx) {
          ptx::tma_load_3d(sbase + C::kDqQ + hx * C::kHalfBytes, &p.tmap_q, bar(QF), hx * 64,
                           it.qt * kTileM, it.b * p.H + it.h, pol);
          ptx::tma_load_3d(sbase + C::kDqDo + hx * C::kHalfBytes, &p.tmap_do, bar(QF), hx * 64,
                           it.qt * kTileM, it.b * p.H + it.h, pol);
        }
        const int kvz = it.b * p.H_kv + it.h / p.group;
        for (int j = 0; j < it.n && ok; ++j) {
          if (entry_cls(it.lst[j], it.t) == kEmpty) continue;
          const int row0 = (int)entry_tile(it.lst[j]) * kTileN;
          // tile g = kv_cnt: K into slot g % KS, V into slot g % VS
          const int ks = (int)(kv_cnt % KS), vs = (int)(kv_cnt % VS);
          if (kv_cnt >= (uint32_t)KS)
            ok = bwait(bar(KE + ks), ((kv_cnt / KS) - 1) & 1, ctl, kBSiteLoad);
          if (!ok) break;
          const uint32_t kdst = sbase + C::kDqK + ks * C::kTileBytes;
          ptx::mbar_arrive_expect_tx(bar(KF + ks), C::kTileBytes);
          for (int hx = 0; hx < C::kHalves; ++hx)
            ptx::tma_load_3d(kdst + hx * C::kHalfBytes, &p.tmap_k, bar(KF + ks), hx * 64, row0,
                             kvz, pol);
          if (kv_cnt >= (uint32_t)VS)
            ok = bwait(bar(VE + vs), ((kv_cnt / VS) - 1) & 1, ctl, kBSiteLoad);
          if (!ok) {
            ++kv_cnt;  // K of this tile is in flight (drained below)
            break;
          }
          const uint32_t vdst = sbase + C::kDqV + vs * C::kTileBytes;
          ptx::mbar_arrive_expect_tx(bar(VF + vs), C::kTileBytes);
          for (int hx = 0; hx < C::kHalves; ++hx)
            ptx::tma_load_3d(vdst + hx * C::kHalfBytes, &p.tmap_v, bar(VF + vs), hx * 64, row0,
                             kvz, pol);
          ++kv_cnt;
          ++v_issued;
        }
        ++act;
      }
      if (!ok) {
        drain_loads(bar(QF), 1, q_issued, p.budget_ns);
        drain_loads(bar(KF), KS, kv_cnt, p.budget_ns);
        drain_loads(bar(VF), VS, v_issued, p.budget_ns);
      }
    }
  } else if (warp == kBMmaWarp) {
    // Tensor Memory: S [0, 128), dP in two buffers [128, 256) and
    // [256, 384) (tile g of the CTA's sequence uses buffer g & 1), dQ
    // [384, 384 + D)
    const uint32_t tS = tmem, tQ = tmem + 384u;
    auto tPb = [&](uint32_t g) { return tmem + 128u + 128u * (g & 1u); };
    const uint64_t q_desc = BDesc<D>::kKMajor + ((sbase + C::kDqQ) >> 4);
    const uint64_t do_desc = BDesc<D>::kKMajor + ((sbase + C::kDqDo) >> 4);
    auto waitw = [&](uint32_t b, uint32_t par) {
      return __all_sync(0xffffffffu, bwait(b, par, ctl, kBSiteMma));
    };
    uint32_t kv_cnt = 0, ds_cnt = 0, scon_cnt = 0;
    int act = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int w = bitem_of(r);
      if (w >= p.n_items) break;
      const It it = item(w);
      if (nonempty(it) == 0) continue;
      if (p.debug_stall == 1) {  // test hook: a wait nothing ever completes
        ok = __all_sync(0xffffffffu, bwait(bar(NEVER), 0, ctl, kBSiteDebugStall + 1));
        if (!ok) break;
      }
      ok = waitw(bar(QF), act & 1);
      if (!ok) break;
      // Software pipeline over the item's key tiles u (tile g = kv0 + u of
      // the CTA's sequence): S(u+1) and dP(u+1) are issued as soon as the
      // elementwise warps have read S(u), dP(u+1) into the other buffer, so
      // both are ready when the elementwise warps finish tile u; dQ(u)
      // follows once dS(u) is written over dP(u)'s buffer (which dP(u+2)
      // overwrites only after dQ(u), in issue order).  V(u) is released
      // after dP(u), K(u) after dQ(u); the K ring is one stage deeper, since
      // S(u+2) follows dQ(u) directly.  Q and dO are released after the
      // item's last S and dP, so the next item's Q loads under this item's
      // last dQ products, and the previous item's dQ must be read out only
      // before this item's first dQ.
      const int m = nonempty(it);
      const uint32_t kv0 = kv_cnt;
      auto kaddr = [&](int u) {
        return sbase + C::kDqK + (uint32_t)(((kv0 + (uint32_t)u) % KS) * C::kTileBytes);
      };
      auto vaddr = [&](int u) {
        return sbase + C::kDqV + (uint32_t)(((kv0 + (uint32_t)u) % VS) * C::kTileBytes);
      };
      auto kv_ready = [&](int u) {
        const uint32_t g = kv0 + (uint32_t)u;
        return waitw(bar(KF + (int)(g % KS)), (g / KS) & 1);
      };
      auto issue_s_dp = [&](int u) -> bool {
        const uint32_t g = kv0 + (uint32_t)u;
        mma_nt<D>(tS, q_desc, BDesc<D>::kKMajor + (kaddr(u) >> 4));  // S = Q K^T
        ptx::mma_commit_elect(bar(SF));
        // V is waited for only now: S does not need it
        if (!waitw(bar(VF + (int)(g % VS)), (g / VS) & 1)) return false;
        ptx::tc_fence_after();
        mma_nt<D>(tPb(g), do_desc, BDesc<D>::kKMajor + (vaddr(u) >> 4));  // dP = dO V^T
        ptx::mma_commit_elect(bar(DPF + (int)(g & 1u)));
        ptx::mma_commit_elect(bar(VE + (int)(g % VS)));
        if (u + 1 == m) ptx::mma_commit_elect(bar(QE));
        return true;
      };
      ok = kv_ready(0);
      if (!ok) break;
      ptx::tc_fence_after();
      ok = issue_s_dp(0);
      if (!ok) break;
      for (int u = 0; u < m && ok; ++u) {
        ok = waitw(bar(SCON), scon_cnt & 1);
        if (!ok) break;
        ++scon_cnt;
        if (u + 1 < m) {
          ok = kv_ready(u + 1);
          if (!ok) break;
          ptx::tc_fence_after();
          ok = issue_s_dp(u + 1);
          if (!ok) break;
        }
        ok = waitw(bar(DSF), ds_cnt & 1);
        if (ok && u == 0 && act > 0) ok = waitw(bar(DQE), (act - 1) & 1);
        if (!ok) break;
        ++ds_cnt;
        ptx::tc_fence_after();
        const uint32_t g = kv0 + (uint32_t)u;
        mma_tn<D>(tQ, tPb(g) + kBPack, BDesc<D>::kMNMajor + (kaddr(u) >> 4), u > 0);  // dQ += dS K
        ptx::mma_commit_elect(bar(KE + (int)(g % KS)));
      }
      kv_cnt = kv0 + (uint32_t)m;
      if (!ok) break;
      ptx::mma_commit_elect(bar(DQF));
      ++act;
    }
    // every MMA done before Tensor Memory is freed
    __syncwarp();
    ptx::mma_commit_elect(bar(DRAIN));
    const uint64_t t0 = ptx::globaltimer_ns();
    bool drained = true;
    while (!ptx::mbar_try_wait(bar(DRAIN), 0)) {
      if (ptx::globaltimer_ns() - t0 > p.budget_ns) {
        drained = false;
        break;
      }
    }
    if (!__all_sync(0xffffffffu, drained) && lane == 0) breport(ctl, ATTN_ERR_TIMEOUT, kBSiteDrain, 0);
  }
  } else {
    // ===================== elementwise: one thread per query row =========
    // half 0: key columns [0, 64) of each tile, half 1: [64, 128); the dQ
    // epilogue splits the D columns the same way
    const int half = warp >> 2, wq = warp & 3;
    const int row = wq * 32 + lane;
    const int cb = kBCols * half;
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t tS = lane_base + (uint32_t)cb, tQ = lane_base + 384u + (uint32_t)(half * D / 2);
    uint32_t s_cnt = 0;
    int act = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int w = bitem_of(r);
      if (w >= p.n_items) break;
      const It it = item(w);
      const int i = it.qt * kTileM + row;
      const bool valid = i < p.S_q;
      const size_t bh = (size_t)it.b * p.H + it.h;
      __nv_bfloat16* dqrow = p.dq + (bh * p.S_q + (size_t)i) * D + half * (D / 2);
      if (nonempty(it) == 0) {
        if (valid) {
          const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < D / 16; ++c) reinterpret_cast<uint4*>(dqrow)[c] = z;
        }
        continue;
      }
      const size_t si = bh * (size_t)p.nQ * kTileM + (size_t)it.qt * kTileM + row;
      const float nlse2 = p.nlse2[si];
      const float ndlt = p.ndelta[si];
      int lo, hi;
      row_keys(p, it.b, i, docs_sorted != 0, lo, hi);
      const bool has_doc = (p.mask_flags & ATTN_MASK_DOCUMENT) != 0 && !docs_sorted;
      const int* doc_b = has_doc ? p.doc_ids + (size_t)it.b * p.S_k : nullptr;
      const int doc_i = (has_doc && valid) ? doc_b[i] : 0;
      const ScoreMod md = make_mod<ALIBI, SOFTCAP>(p, it.h);
      const int qpos = i + p.q_offset;
      for (int j = 0; j < it.n && ok; ++j) {
        const uint32_t cls = entry_cls(it.lst[j], it.t);
        if (cls == kEmpty) continue;
        const int j0 = (int)entry_tile(it.lst[j]) * kTileN + cb;  // first key of this half
        const uint32_t g = s_cnt;  // this tile's place in the CTA's sequence
        // its dP buffer: this half's columns, and where dS is packed
        const uint32_t tP = lane_base + 128u + 128u * (g & 1u) + (uint32_t)cb,
                       tPk = lane_base + 128u + 128u * (g & 1u) + kBPack + 32u * (uint32_t)half;
        {
          const bool got = bwait(bar(SF), s_cnt & 1, ctl, kBSiteElem);
          ok = __all_sync(0xffffffffu, got);
          if (!ok) break;
        }
        ++s_cnt;
        ptx::tc_fence_after();
        // this half of S into registers, then release it for S(u+1); the
        // modified scores, then the mask in a loop of its own (a branch per
        // element would split the unrolled loop and serialise the
        // exponentials)
        float tv[kBCols];
        {
          uint32_t ra[32], rb[32];
          ptx::tmem_ld32(tS, ra);
          ptx::tmem_ld32(tS + 32u, rb);
          ptx::tmem_wait_ld();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(SCON));
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            tv[c] = __uint_as_float(ra[c]);
            tv[32 + c] = __uint_as_float(rb[c]);
          }
        }
        // the plain score (a scale) is folded into the exponential below
        constexpr bool kPlain = !ALIBI && !SOFTCAP;
        add_rel_bias<ALIBI, SOFTCAP, kBCols>(tv, p, it.h, j0 - qpos, 1, md);
        if constexpr (!kPlain) score_cols<ALIBI, SOFTCAP>(tv, (float)(j0 - qpos), 1.0f, md, p);
        if (cls == kPartial) {
          const int clo = lo - j0, chi = hi - j0;
          if (has_doc) {
#pragma unroll
            for (int c = 0; c < kBCols; ++c) {
              const int jj = j0 + c;
              const bool vis = (c >= clo) & (c <= chi) & (jj < p.S_k) &&
                               doc_b[jj < p.S_k ? jj : 0] == doc_i;
              tv[c] = vis ? tv[c] : -INFINITY;
            }
          } else {
#pragma unroll
            for (int c = 0; c < kBCols; ++c) tv[c] = ((c >= clo) & (c <= chi)) ? tv[c] : -INFINITY;
          }
        }
        // P (times the soft cap's derivative), in place, while dP computes;
        // two columns per paired fp32 instruction (a masked -inf stays -inf:
        // the scale is positive)
        {
          const uint64_t sc2 = ptx::f2(kPlain ? md.sc : 1.0f, kPlain ? md.sc : 1.0f),
                         nl2 = ptx::f2(nlse2, nlse2);
#pragma unroll
          for (int c = 0; c < kBCols; c += 2) {
            float xa, xb;
            ptx::f2_split(ptx::ffma2(ptx::f2(tv[c], tv[c + 1]), sc2, nl2), xa, xb);
            float pa = ptx::ex2_approx(xa), pb = ptx::ex2_approx(xb);
            if constexpr (SOFTCAP) {  // masked: t = -inf, clamped so the factor is 0
              const float ua = fmaxf(tv[c], -md.capl2) * md.inv_capl2;
              const float ub = fmaxf(tv[c + 1], -md.capl2) * md.inv_capl2;
              pa *= 1.0f - ua * ua;
              pb *= 1.0f - ub * ub;
            }
            tv[c] = pa;
            tv[c + 1] = pb;
          }
        }
        {
          const bool got = bwait(bar(DPF + (int)(g & 1u)), (g >> 1) & 1u, ctl, kBSiteElem);
          ok = __all_sync(0xffffffffu, got);
          if (!ok) break;
        }
        ptx::tc_fence_after();
        // dS = P (dP - Delta): this half's 64 columns of dP, then 32 packed
        // columns over them (paired fp32: dP + (-Delta), then times P)
        {
          uint32_t d0[32], d1[32], pk[32];
          ptx::tmem_ld32(tP, d0);
          ptx::tmem_ld32(tP + 32u, d1);
          ptx::tmem_wait_ld();
          const uint64_t nd2 = ptx::f2(ndlt, ndlt);
          auto ds2 = [&](uint32_t a, uint32_t b, int c) {
            float x, y;
            ptx::f2_split(ptx::fmul2(ptx::fadd2(ptx::f2(__uint_as_float(a), __uint_as_float(b)),
                                                nd2),
                                     ptx::f2(tv[c], tv[c + 1])),
                          x, y);
            return ptx::pack_bf16x2(x, y);
          };
#pragma unroll
          for (int c2 = 0; c2 < 16; ++c2) {
            pk[c2] = ds2(d0[2 * c2], d0[2 * c2 + 1], 2 * c2);
            pk[16 + c2] = ds2(d1[2 * c2], d1[2 * c2 + 1], 32 + 2 * c2);
          }
          ptx::tmem_st32(tPk, pk);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(DSF));
      }
      if (!ok) break;
      {
        const bool got = bwait(bar(DQF), act & 1, ctl, kBSiteElem);
        ok = __all_sync(0xffffffffu, got);
        if (!ok) break;
      }
      ptx::tc_fence_after();
      {
        // every load in flight before one wait; dQ's columns are free for the
        // next item as soon as they have landed
        uint32_t o[D / 64][32];
#pragma unroll
        for (int c4 = 0; c4 < D / 64; ++c4) ptx::tmem_ld32(tQ + (uint32_t)(c4 * 32), o[c4]);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(DQE));
        if (valid) {
          const bool al32 = (reinterpret_cast<uintptr_t>(p.dq) & 31u) == 0;
#pragma unroll
          for (int c4 = 0; c4 < D / 64; ++c4) {
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 16; ++c)
              pk[c] = ptx::pack_bf16x2(__uint_as_float(o[c4][2 * c]) * p.scale,
                                       __uint_as_float(o[c4][2 * c + 1]) * p.scale);
            store_row32(dqrow + c4 * 32, pk, al32);
          }
        }
      }
      ++act;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kBMmaWarp) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kBTmemCols);
  }
}

// ---------------------------------------------------------------- dK dV ---
template <int D, bool ALIBI, bool SOFTCAP>
__global__ void __launch_bounds__(kBThreads, 1) bwd_dkdv_kernel(const __grid_constant__ BParams p) {
  using C = BCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  ptx::griddep_wait();
  const int docs_sorted = p.hdr->docs_sorted;

  auto bar = [&](int i) { return sbase + (uint32_t)(C::kKvBar + 8 * i); };
  enum { KF = 0, KE = 1, QF = 2, QE = 4, SF = 6, PF = 7, AF = 8, AE = 9, DRAIN = 10, DPF = 11,
         DSF = 12, NEVER = 13 };
  static_assert(NEVER < C::kNumBars, "barrier slots");
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::kKvBar + 8 * C::kNumBars);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::kKvBar + 8 * C::kNumBars + 4);
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(KF), 1);
    ptx::mbar_init(bar(KE), 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(bar(QF + s), 1);
      ptx::mbar_init(bar(QE + s), 1);
    }
    // one arrival per elementwise warp
    ptx::mbar_init(bar(SF), 1);
    ptx::mbar_init(bar(PF), 8);
    ptx::mbar_init(bar(AF), 1);
    ptx::mbar_init(bar(AE), 8);
    ptx::mbar_init(bar(DPF), 1);
    ptx::mbar_init(bar(DSF), 8);
    ptx::mbar_init(bar(DRAIN), 1);
    ptx::mbar_init(bar(NEVER), 1);  // the test hook's: nothing arrives on it
    *s_abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kBMmaWarp) {
    ptx::tmem_alloc(ptx::smem_addr(s_tmem), kBTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const BCtl ctl{s_abort, sbase + (uint32_t)(C::kKvBar + 8 * C::kNumBars + 4), p.status,
                 p.budget_ns};

  // Item w -> (b, K/V head, key tile); its work units are (query head of the
  // group, query tile of the transposed list).
  struct It {
    int b, hk, kt, n;
    const uint32_t* lst;
  };
  auto item = [&](int w) {
    It it;
    it.kt = w % p.nK;
    const int bh = w / p.nK;
    it.b = bh / p.H_kv;
    it.hk = bh % p.H_kv;
    const int e = (p.bm == 1 ? 0 : it.b) * p.nK + it.kt;
    it.n = p.cnt_t[e];
    it.lst = p.list_t + (size_t)e * p.nQ;
    return it;
  };
  auto stage_addr = [&](int st) { return sbase + (uint32_t)(C::kKvStage0 + st * C::kKvStageBytes); };

  if (warp >= 8) {
  if (warp == kBLoadWarp) {
    if (lane == 0) {
      ptx::prefetch_tmap(&p.tmap_q);
      ptx::prefetch_tmap(&p.tmap_do);
      ptx::prefetch_tmap(&p.tmap_k);
      ptx::prefetch_tmap(&p.tmap_v);
      const uint64_t pol = ptx::policy_evict_last();
      uint32_t q_cnt = 0, k_issued = 0;
      int act = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int w = bitem_of(r);
        if (w >= p.n_items) break;
        const It it = item(w);
        if (it.n == 0) continue;
        if (act > 0) ok = bwait(bar(KE), (act - 1) & 1, ctl, kBSiteLoad);
        if (!ok) break;
        const int kvz = it.b * p.H_kv + it.hk;
        ptx::mbar_arrive_expect_tx(bar(KF), 2 * C::kTileBytes);
        k_issued = act + 1;
        for (int hx = 0; hx < C::kHalves; ++hx) {
          ptx::tma_load_3d(sbase + C::kKvK + hx * C::kHalfBytes, &p.tmap_k, bar(KF), hx * 64,
                           it.kt * kTileN, kvz, pol);
          ptx::tma_load_3d(sbase + C::kKvV + hx * C::kHalfBytes, &p.tmap_v, bar(KF), hx * 64,
                           it.kt * kTileN, kvz, pol);
        }
        for (int g = 0; g < p.group && ok; ++g) {
          const int h = it.hk * p.group + g;
          const size_t bh = (size_t)it.b * p.H + h;
          for (int u = 0; u < it.n && ok; ++u) {
            const int qt = (int)entry_tile(it.lst[u]);
            const int st = (int)(q_cnt & 1);
            if (q_cnt >= 2) ok = bwait(bar(QE + st), ((q_cnt >> 1) - 1) & 1, ctl, kBSiteLoad);
            if (!ok) break;
            const uint32_t dst = stage_addr(st);
            ptx::mbar_arrive_expect_tx(bar(QF + st), 2 * C::kTileBytes + 2 * kTileM * 4);
            for (int hx = 0; hx < C::kHalves; ++hx) {
              ptx::tma_load_3d(dst + hx * C::kHalfBytes, &p.tmap_q, bar(QF + st), hx * 64,
                               qt * kTileM, (int)bh, pol);
              ptx::tma_load_3d(dst + C::kTileBytes + hx * C::kHalfBytes, &p.tmap_do, bar(QF + st),
                               hx * 64, qt * kTileM, (int)bh, pol);
            }
            const size_t so = bh * (size_t)p.nQ * kTileM + (size_t)qt * kTileM;
            ptx::bulk_load(dst + 2 * C::kTileBytes, p.nlse2 + so, kTileM * 4, bar(QF + st));
            ptx::bulk_load(dst + 2 * C::kTileBytes + kTileM * 4, p.ndelta + so, kTileM * 4,
                           bar(QF + st));
            ++q_cnt;
          }
        }
        ++act;
      }
      if (!ok) {
        drain_loads(bar(KF), 1, k_issued, p.budget_ns);
        drain_loads(bar(QF), 2, q_cnt, p.budget_ns);
      }
    }
  } else if (warp == kBMmaWarp) {
    const uint32_t tST = tmem, tDPT = tmem + 128u, tDV = tmem + 256u, tDK = tmem + 256u + D;
    const uint64_t k_kmaj = BDesc<D>::kKMajor + ((sbase + C::kKvK) >> 4);
    const uint64_t v_kmaj = BDesc<D>::kKMajor + ((sbase + C::kKvV) >> 4);
    auto waitw = [&](uint32_t b, uint32_t par) {
      return __all_sync(0xffffffffu, bwait(b, par, ctl, kBSiteMma));
    };
    uint32_t q_cnt = 0, p_cnt = 0, ds_cnt = 0;
    int act = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int w = bitem_of(r);
      if (w >= p.n_items) break;
      const It it = item(w);
      if (it.n == 0) continue;
      if (p.debug_stall == 2) {  // test hook: a wait nothing ever completes
        ok = __all_sync(0xffffffffu, bwait(bar(NEVER), 0, ctl, kBSiteDebugStall + 2));
        if (!ok) break;
      }
      ok = waitw(bar(KF), act & 1);
      if (ok && act > 0) ok = waitw(bar(AE), (act - 1) & 1);
      if (!ok) break;
      // Software pipeline over the item's units u: dV(u) starts as soon as
      // P^T(u) is written, S^T(u+1) follows it (P^T(u) has been read), and
      // dK(u) waits for dS^T(u), so the elementwise warps' next tile is
      // computed while dK(u) and dP^T(u+1) run.
      const int units = p.group * it.n;
      const uint32_t q0 = q_cnt;
      auto qaddr = [&](int u) { return stage_addr((int)((q0 + (uint32_t)u) & 1)); };
      auto q_ready = [&](int u) {
        return waitw(bar(QF + (int)((q0 + (uint32_t)u) & 1)), ((q0 + (uint32_t)u) >> 1) & 1);
      };
      ok = q_ready(0);
      if (!ok) break;
      ptx::tc_fence_after();
      mma_nt<D>(tST, k_kmaj, BDesc<D>::kKMajor + (qaddr(0) >> 4));  // S^T = K Q^T
      ptx::mma_commit_elect(bar(SF));
      mma_nt<D>(tDPT, v_kmaj, BDesc<D>::kKMajor + ((qaddr(0) + C::kTileBytes) >> 4));  // dP^T
      ptx::mma_commit_elect(bar(DPF));
      for (int u = 0; u < units && ok; ++u) {
        ok = waitw(bar(PF), p_cnt & 1);
        if (!ok) break;
        ++p_cnt;
        ptx::tc_fence_after();
        mma_tn<D>(tDV, tST + kBPack, BDesc<D>::kMNMajor + ((qaddr(u) + C::kTileBytes) >> 4),
                  u > 0);  // dV += P^T dO
        if (u + 1 < units) {
          ok = q_ready(u + 1);
          if (!ok) break;
          ptx::tc_fence_after();
          mma_nt<D>(tST, k_kmaj, BDesc<D>::kKMajor + (qaddr(u + 1) >> 4));
          ptx::mma_commit_elect(bar(SF));
        }
        ok = waitw(bar(DSF), ds_cnt & 1);
        if (!ok) break;
        ++ds_cnt;
        ptx::tc_fence_after();
        mma_tn<D>(tDK, tDPT + kBPack, BDesc<D>::kMNMajor + (qaddr(u) >> 4), u > 0);  // dK += dS^T Q
        ptx::mma_commit_elect(bar(QE + (int)((q0 + (uint32_t)u) & 1)));
        if (u + 1 < units) {
          mma_nt<D>(tDPT, v_kmaj, BDesc<D>::kKMajor + ((qaddr(u + 1) + C::kTileBytes) >> 4));
          ptx::mma_commit_elect(bar(DPF));
        }
      }
      q_cnt = q0 + (uint32_t)units;
      if (!ok) break;
      ptx::mma_commit_elect(bar(AF));
      ptx::mma_commit_elect(bar(KE));
      ++act;
    }
    __syncwarp();
    ptx::mma_commit_elect(bar(DRAIN));
    const uint64_t t0 = ptx::globaltimer_ns();
    bool drained = true;
    while (!ptx::mbar_try_wait(bar(DRAIN), 0)) {
      if (ptx::globaltimer_ns() - t0 > p.budget_ns) {
        drained = false;
        break;
      }
    }
    if (!__all_sync(0xffffffffu, drained) && lane == 0) breport(ctl, ATTN_ERR_TIMEOUT, kBSiteDrain, 0);
  }
  } else {
    // ===================== elementwise: one thread per key ================
    // half 0: query columns [0, 64) of each tile, half 1: [64, 128); the
    // dK / dV epilogue splits the D columns the same way
    const int half = warp >> 2, wq = warp & 3;
    const int row = wq * 32 + lane;
    const int cb = kBCols * half;
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t tST = lane_base + (uint32_t)cb, tDPT = lane_base + 128u + (uint32_t)cb,
                   tPk = lane_base + kBPack + 32u * (uint32_t)half,
                   tDSk = lane_base + 128u + kBPack + 32u * (uint32_t)half,
                   tDV = lane_base + 256u + (uint32_t)(half * D / 2),
                   tDK = lane_base + 256u + D + (uint32_t)(half * D / 2);
    uint32_t q_cnt = 0;
    int act = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int w = bitem_of(r);
      if (w >= p.n_items) break;
      const It it = item(w);
      const int j = it.kt * kTileN + row;  // this thread's key
      const bool valid = j < p.S_k;
      const size_t kvh = (size_t)it.b * p.H_kv + it.hk;
      __nv_bfloat16* dkrow = p.dk + (kvh * p.S_k + (size_t)j) * D + half * (D / 2);
      __nv_bfloat16* dvrow = p.dv + (kvh * p.S_k + (size_t)j) * D + half * (D / 2);
      if (it.n == 0) {
        if (valid) {
          const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            reinterpret_cast<uint4*>(dkrow)[c] = z;
            reinterpret_cast<uint4*>(dvrow)[c] = z;
          }
        }
        continue;
      }
      int ilo, ihi;
      key_rows(p, it.b, j, docs_sorted != 0, ilo, ihi);
      const bool has_doc = (p.mask_flags & ATTN_MASK_DOCUMENT) != 0 && !docs_sorted;
      const int* doc_b = has_doc ? p.doc_ids + (size_t)it.b * p.S_k : nullptr;
      const int doc_j = (has_doc && valid) ? doc_b[j] : 0;
      for (int g = 0; g < p.group && ok; ++g) {
        const int h = it.hk * p.group + g;
        const ScoreMod md = make_mod<ALIBI, SOFTCAP>(p, h);
        for (int u = 0; u < it.n && ok; ++u) {
          const uint32_t cls = entry_cls(it.lst[u], 0);
          const int i0 = (int)entry_tile(it.lst[u]) * kTileM + cb;  // first query of this half
          const int st = (int)(q_cnt & 1);
          {
            const bool got = bwait(bar(SF), q_cnt & 1, ctl, kBSiteElem);
            ok = __all_sync(0xffffffffu, got);
            if (!ok) break;
          }
          ptx::tc_fence_after();
          // -LSE (log2 units) and -Delta of this half's 64 queries in shared
          // memory
          const uint32_t s_nlse2 = sbase + (uint32_t)(C::kKvStage0 + st * C::kKvStageBytes +
                                                      2 * C::kTileBytes + 4 * cb);
          const uint32_t s_ndelta = s_nlse2 + 4u * kTileM;
          // this half of S^T (this key against 64 queries) into registers
          float tv[kBCols];
          const float jb = (float)(j - (i0 + p.q_offset));  // bias position of column 0
          {
            uint32_t ra[32], rb[32];
            ptx::tmem_ld32(tST, ra);
            ptx::tmem_ld32(tST + 32u, rb);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              tv[c] = __uint_as_float(ra[c]);
              tv[32 + c] = __uint_as_float(rb[c]);
            }
          }
          // the plain score (a scale) is folded into the exponential below
          constexpr bool kPlain = !ALIBI && !SOFTCAP;
          add_rel_bias<ALIBI, SOFTCAP, kBCols>(tv, p, h, j - (i0 + p.q_offset), -1, md);
          if constexpr (!kPlain) score_cols<ALIBI, SOFTCAP>(tv, jb, -1.0f, md, p);
          // the mask in a loop of its own (rows beyond S_k see nothing)
          if (!valid || cls == kPartial) {
            const int clo = ilo - i0, chi = ihi - i0;
            if (has_doc) {
#pragma unroll
              for (int c = 0; c < kBCols; ++c) {
                const int qi = i0 + c;
                const bool vis = valid & (c >= clo) & (c <= chi) & (qi < p.S_q) &&
                                 doc_b[qi < p.S_q ? qi : 0] == doc_j;
                tv[c] = vis ? tv[c] : -INFINITY;
              }
            } else {
#pragma unroll
              for (int c = 0; c < kBCols; ++c)
                tv[c] = (valid & (c >= clo) & (c <= chi)) ? tv[c] : -INFINITY;
            }
          }
          // P^T, packed over this half's S^T columns for dV; kept (times the
          // soft cap's derivative) in place for dS^T.  -LSE of the 64 queries
          // comes in 16-byte shared-memory loads (the same address for every
          // lane); two columns per paired fp32 instruction (a masked -inf
          // stays -inf: the scale is positive).
          {
            uint32_t pp[32];
            const uint64_t sc2 = ptx::f2(kPlain ? md.sc : 1.0f, kPlain ? md.sc : 1.0f);
#pragma unroll
            for (int c4 = 0; c4 < kBCols / 4; ++c4) {
              const float4 lv = ptx::lds_v4(s_nlse2 + 16u * (uint32_t)c4);
              const float lq[4] = {lv.x, lv.y, lv.z, lv.w};
#pragma unroll
              for (int e = 0; e < 4; e += 2) {
                const int c = 4 * c4 + e;
                float xa, xb;
                ptx::f2_split(ptx::ffma2(ptx::f2(tv[c], tv[c + 1]), sc2, ptx::f2(lq[e], lq[e + 1])),
                              xa, xb);
                const float pa = ptx::ex2_approx(xa), pb = ptx::ex2_approx(xb);
                float da = 1.0f, db = 1.0f;
                if constexpr (SOFTCAP) {
                  const float ua = fmaxf(tv[c], -md.capl2) * md.inv_capl2;
                  const float ub = fmaxf(tv[c + 1], -md.capl2) * md.inv_capl2;
                  da = 1.0f - ua * ua;
                  db = 1.0f - ub * ub;
                }
                tv[c] = pa * da;
                tv[c + 1] = pb * db;
                pp[2 * c4 + e / 2] = ptx::pack_bf16x2(pa, pb);
              }
            }
            ptx::tmem_st32(tPk, pp);
          }
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(PF));
          {
            const bool got = bwait(bar(DPF), q_cnt & 1, ctl, kBSiteElem);
            ok = __all_sync(0xffffffffu, got);
            if (!ok) break;
          }
          ptx::tc_fence_after();
          // dS^T = P^T (dP^T - Delta): this half's 64 columns of dP^T, then
          // 32 packed columns over them
          {
            uint32_t d0[32], d1[32], pk[32];
            ptx::tmem_ld32(tDPT, d0);
            ptx::tmem_ld32(tDPT + 32u, d1);
            ptx::tmem_wait_ld();
            // paired fp32: dP^T + (-Delta), then times P^T
            auto ds2 = [&](uint32_t x0, uint32_t x1, float n0, float n1, int c) {
              float x, y;
              ptx::f2_split(
                  ptx::fmul2(ptx::fadd2(ptx::f2(__uint_as_float(x0), __uint_as_float(x1)),
                                        ptx::f2(n0, n1)),
                             ptx::f2(tv[c], tv[c + 1])),
                  x, y);
              return ptx::pack_bf16x2(x, y);
            };
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              const float4 a = ptx::lds_v4(s_ndelta + 16u * (uint32_t)c4),
                           b = ptx::lds_v4(s_ndelta + 16u * (uint32_t)(8 + c4));
              const int c = 4 * c4;
              pk[2 * c4] = ds2(d0[c], d0[c + 1], a.x, a.y, c);
              pk[2 * c4 + 1] = ds2(d0[c + 2], d0[c + 3], a.z, a.w, c + 2);
              pk[16 + 2 * c4] = ds2(d1[c], d1[c + 1], b.x, b.y, 32 + c);
              pk[17 + 2 * c4] = ds2(d1[c + 2], d1[c + 3], b.z, b.w, 34 + c);
            }
            ptx::tmem_st32(tDSk, pk);
          }
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(DSF));
          ++q_cnt;
        }
      }
      if (!ok) break;
      {
        const bool got = bwait(bar(AF), act & 1, ctl, kBSiteElem);
        ok = __all_sync(0xffffffffu, got);
        if (!ok) break;
      }
      ptx::tc_fence_after();
      {
        // every load in flight before one wait; the accumulators are free
        // for the next item as soon as they have landed
        uint32_t ov[D / 64][32], ok32[D / 64][32];
#pragma unroll
        for (int c4 = 0; c4 < D / 64; ++c4) {
          ptx::tmem_ld32(tDV + (uint32_t)(c4 * 32), ov[c4]);
          ptx::tmem_ld32(tDK + (uint32_t)(c4 * 32), ok32[c4]);
        }
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar(AE));
        if (valid) {
          const uintptr_t kv_bits =
              reinterpret_cast<uintptr_t>(p.dk) | reinterpret_cast<uintptr_t>(p.dv);
          const bool al32 = (kv_bits & 31u) == 0;
#pragma unroll
          for (int c4 = 0; c4 < D / 64; ++c4) {
            uint32_t pv[16], pkk[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              pv[c] = ptx::pack_bf16x2(__uint_as_float(ov[c4][2 * c]),
                                       __uint_as_float(ov[c4][2 * c + 1]));
              pkk[c] = ptx::pack_bf16x2(__uint_as_float(ok32[c4][2 * c]) * p.scale,
                                        __uint_as_float(ok32[c4][2 * c + 1]) * p.scale);
            }
            store_row32(dvrow + c4 * 32, pv, al32);
            store_row32(dkrow + c4 * 32, pkk, al32);
          }
        }
      }
      ++act;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kBMmaWarp) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kBTmemCols);
  }
}

// ---------------------------------------------------------------- host ----

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn bget_encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// [outer][S][D] bf16 as 3-D (D, S, outer); box 64 x 128 x 1, 128-byte
// swizzle; rows beyond S read as zero.
bool bmake_map(CUtensorMap* map, const void* ptr, int D, int S, int outer) {
  EncodeTiledFn enc = bget_encode_tiled();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)outer};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)S * (cuuint64_t)D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)kTileM, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The opt-in shared memory size is a function attribute: it is set once per
// device and kernel (attr_set: that kernel's flag for this device, or null
// to set it on every call).  A concurrent first call repeats the same
// idempotent call.
constexpr int kBLaunchCacheDevices = 64;

template <typename K>
cudaError_t launch_ex(K kern, int grid, int smem, cudaStream_t stream, const BParams& bp,
                      std::atomic<bool>* attr_set) {
  if (attr_set == nullptr || !attr_set->load(std::memory_order_relaxed)) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (attr_set != nullptr) attr_set->store(true, std::memory_order_relaxed);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kBThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, bp);
}

template <int D, bool ALIBI, bool SOFTCAP>
cudaError_t launch_bwd_variant(BParams bp, int sms, cudaStream_t s, int dev) {
  using C = BCfg<D>;
  static std::atomic<bool> set_dq[kBLaunchCacheDevices], set_kv[kBLaunchCacheDevices];
  const bool cache = dev >= 0 && dev < kBLaunchCacheDevices;
  bp.n_items = bp.B * bp.H * bp.nQ;
  const int g1 = bp.n_items < sms ? bp.n_items : sms;
  cudaError_t err = launch_ex(bwd_dq_kernel<D, ALIBI, SOFTCAP>, g1 > 0 ? g1 : 1, C::kSmemAllocDq,
                              s, bp, cache ? &set_dq[dev] : nullptr);
  if (err != cudaSuccess) return err;
  bp.n_items = bp.B * bp.H_kv * bp.nK;
  const int g2 = bp.n_items < sms ? bp.n_items : sms;
  return launch_ex(bwd_dkdv_kernel<D, ALIBI, SOFTCAP>, g2 > 0 ? g2 : 1, C::kSmemAllocKv, s, bp,
                   cache ? &set_kv[dev] : nullptr);
}

template <int D>
cudaError_t launch_bwd_d(const BParams& bp, bool alibi, bool softcap, int sms, cudaStream_t s,
                         int dev) {
  if (alibi && softcap) return launch_bwd_variant<D, true, true>(bp, sms, s, dev);
  if (alibi) return launch_bwd_variant<D, true, false>(bp, sms, s, dev);
  if (softcap) return launch_bwd_variant<D, false, true>(bp, sms, s, dev);
  return launch_bwd_variant<D, false, false>(bp, sms, s, dev);
}

}  // namespace

cudaError_t launch_attn_bwd(const BwdArgs& a, cudaStream_t stream) {
  BParams bp;
  memset(&bp, 0, sizeof(bp));
  if (!bmake_map(&bp.tmap_q, a.q, a.D, a.S_q, a.B * a.H) ||
      !bmake_map(&bp.tmap_do, a.dout, a.D, a.S_q, a.B * a.H) ||
      !bmake_map(&bp.tmap_k, a.k, a.D, a.S_k, a.B * a.H_kv) ||
      !bmake_map(&bp.tmap_v, a.v, a.D, a.S_k, a.B * a.H_kv))
    return cudaErrorInvalidValue;
  const BlockMaskGeom g = block_mask_geom(a.B, a.S_q, a.S_k, a.mask.flags);
  const BlockMaskTGeom gt = block_mask_t_geom(a.B, a.S_q, a.S_k, a.mask.flags);
  bp.dq = reinterpret_cast<__nv_bfloat16*>(a.dq);
  bp.dk = reinterpret_cast<__nv_bfloat16*>(a.dk);
  bp.dv = reinterpret_cast<__nv_bfloat16*>(a.dv);
  const size_t padded = (size_t)a.B * a.H * (size_t)g.nQ * kTileM;
  bp.nlse2 = a.rowstat;
  bp.ndelta = a.rowstat + padded;
  bp.B = a.B;
  bp.H = a.H;
  bp.H_kv = a.H_kv;
  bp.S_q = a.S_q;
  bp.S_k = a.S_k;
  bp.group = a.H / a.H_kv;
  bp.nQ = g.nQ;
  bp.nK = g.nK;
  bp.nP = g.nP;
  bp.bm = g.bm;
  bp.scale = a.scale;
  bp.scale_log2 = a.scale * kBLog2e;
  bp.softcap = (a.score_flags & ATTN_SCORE_SOFTCAP) ? a.softcap : 0.f;
  bp.mask_flags = a.mask.flags;
  bp.window = a.mask.window;
  bp.q_offset = a.mask.q_offset;
  bp.doc_ids = a.mask.doc_ids;
  bp.prefix_len = a.mask.prefix_len;
  bp.alibi_slopes = a.alibi_slopes;
  bp.alibi_on = (a.score_flags & ATTN_SCORE_ALIBI) ? 1 : 0;
  bp.rel_bias = (a.score_flags & ATTN_SCORE_RELBIAS) ? a.rel_bias : nullptr;
  bp.rel_max = a.rel_max;
  const char* base = reinterpret_cast<const char*>(a.block_mask);
  bp.hdr = reinterpret_cast<const BlockMaskHeader*>(base);
  bp.cnt = reinterpret_cast<const int32_t*>(base + g.cnt_off);
  bp.list = reinterpret_cast<const uint32_t*>(base + g.list_off);
  if (g.doc_off != 0) {
    bp.doc_lo = reinterpret_cast<const int32_t*>(base + g.doc_off);
    bp.doc_hi = bp.doc_lo + (size_t)g.bm * a.S_k;
  }
  const char* tb = reinterpret_cast<const char*>(a.block_mask_t);
  bp.cnt_t = reinterpret_cast<const int32_t*>(tb);
  bp.list_t = reinterpret_cast<const uint32_t*>(tb + gt.list_off);
  bp.status = a.status;
  const double ms = a.wait_budget_ms > 0 ? a.wait_budget_ms : 2000.0;
  bp.budget_ns = (uint64_t)(ms * 1e6);
  bp.debug_stall = a.debug_stall;
  bp.tlim = -1.0f;  // no polynomial unless its coefficients are normal numbers
  if (bp.softcap > 0.f) {
    // the score reaches the cap as y = 2 log2(e) x / cap = 2 log2(e) u
    const double l2e = 1.4426950408889634, kk = 1.0 / (2.0 * l2e);
    const double C = (double)bp.softcap * l2e;
    const double r[3] = {ATTN_TANH_POLY_R0, ATTN_TANH_POLY_R1, ATTN_TANH_POLY_R2};
    double kpow = kk;
    bool normal = true;
    for (int i = 0; i < 3; ++i) {
      bp.tq[i] = (float)(C * r[i] * kpow);
      normal = normal && fabsf(bp.tq[i]) >= FLT_MIN && isfinite(bp.tq[i]);
      kpow *= kk * kk;
    }
    if (normal) bp.tlim = (float)(ATTN_TANH_POLY_U0 / kk);
  }

  // row statistics, then the two gradient kernels
  const int BH = a.B * a.H;
  const long long rows = (long long)padded;
  const unsigned blocks = (unsigned)((rows + kPrepRows - 1) / kPrepRows);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const __nv_bfloat16* o = reinterpret_cast<const __nv_bfloat16*>(a.out);
  const __nv_bfloat16* dout = reinterpret_cast<const __nv_bfloat16*>(a.dout);
  cudaError_t err = (a.D == 64)
                        ? cudaLaunchKernelEx(&cfg, bwd_prep_kernel<64>, o, dout, a.lse, a.rowstat,
                                             a.rowstat + padded, BH, a.S_q, g.nQ)
                        : cudaLaunchKernelEx(&cfg, bwd_prep_kernel<128>, o, dout, a.lse,
                                             a.rowstat, a.rowstat + padded, BH, a.S_q, g.nQ);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorUnknown;
  static std::atomic<int> sm_count[kBLaunchCacheDevices];
  const bool cache = dev >= 0 && dev < kBLaunchCacheDevices;
  if (cache) sms = sm_count[dev].load(std::memory_order_relaxed);
  if (sms == 0) {
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return cudaErrorUnknown;
    if (cache) sm_count[dev].store(sms, std::memory_order_relaxed);
  }
  const bool alibi = (a.score_flags & (ATTN_SCORE_ALIBI | ATTN_SCORE_RELBIAS)) != 0;
  const bool softcap = (a.score_flags & ATTN_SCORE_SOFTCAP) != 0;
  if (a.D == 64) return launch_bwd_d<64>(bp, alibi, softcap, sms, stream, dev);
  return launch_bwd_d<128>(bp, alibi, softcap, sms, stream, dev);
}

}  // namespace attn
