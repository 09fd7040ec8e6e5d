// attn_fwd_sm103.cu -- fused attention forward for GB300 (sm_103a).
//
// One persistent CTA per SM walks a list of work items; an item is a pair of
// 128-row query tiles of one (batch, head).  Warp roles:
//
//   warps 0-3  softmax warpgroup for query tile 0 (one thread per row)
//   warps 4-7  softmax warpgroup for query tile 1
//   warp  8    TMA producer: a ring of K / V tiles
//   warp  9    Tensor Memory owner; MMA issuer for query tile 0
//   warp 10    MMA issuer for query tile 1
//   warp 11    TMA producer: Q tiles
//
// Per key tile j the tensor core computes S_t = Q_t K_j^T into Tensor Memory
// (fp32), the softmax warpgroup of tile t turns S_t into P_t (bf16, written
// back over S_t in Tensor Memory) and the tensor core accumulates
// O_t += P_t V_j in Tensor Memory.  The two query tiles alternate so that
// one tile's softmax overlaps the other tile's MMAs ("FlashAttention-4
// explained", "Forward pass fixes", "Ping-pong scheduling").  The output
// accumulator is rescaled only when the running row max grows by more than
// a threshold ("Conditional rescaling").  The score matrix never leaves the
// SM ("Enter Tri Dao and FlashAttention").
//
// Each query tile has its own issuing thread with the chain
//   S_t(j), [P_t(j) ready] PV_t(j), S_t(j+1), ...
// and the tensor pipe interleaves the two chains, so each softmax
// warpgroup hides behind the other tile's MMAs.  S_t(j+1) overwrites the
// Tensor Memory that P_t(j) occupies; it is issued after PV_t(j) by the same
// thread and tcgen05 MMAs execute in issue order.
//
// CTA-pair form (PAIR, D = 128; "FlashAttention-4 explained", "TMEM and
// 2-CTA MMA", "2-CTA MMA mode"): two CTAs of a cluster share one work item
// of four query tiles; CTA r holds query tiles 2t + r of it.  Every S and PV
// product of tile t is one tcgen05 MMA with M = 256 (cta_group::2) issued by
// rank 0, which reads each CTA's own Q rows (or P in Tensor Memory) and half
// of the key / value tile from each CTA's shared memory: keys
// [64 r, 64 r + 64) of K, columns [64 r, 64 r + 64) of V.  Each CTA thus
// stages half of every K/V tile, the per-SM shared-memory traffic of the B
// operand halves, and one K/V tile serves 512 query rows.  The softmax is
// unchanged: each CTA's accumulators hold its own 128 rows.  Shared
// barriers (operands landed, P ready, O free) live in rank 0, the rest in
// both CTAs, signalled by multicast commits.
//
// Every mbarrier wait is bounded by a time budget; on expiry the kernel
// records ATTN_ERR_TIMEOUT in the device status word (and raises the abort
// flag of both CTAs of a pair), drains its own in-flight copies and MMAs,
// frees Tensor Memory and returns.
#include <atomic>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <float.h>
#include <math.h>

#include <type_traits>

#include "attn_internal.h"
#include "sm103_ptx.cuh"
#include "tanh_poly.h"

namespace attn {

namespace {

// Three warpgroups: two softmax warpgroups and one producer warpgroup whose
// warp 8 loads K/V, warps 9 and 10 issue MMAs and warp 11 loads Q.  384 threads launch with 168
// registers each; the producer warpgroup drops to kRegsProducer and the
// softmax warpgroups grow to kRegsSoftmax, which uses the same total:
// 256 * 216 + 128 * 72 = 384 * 168.
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kQLoadWarp = 11;
constexpr int kThreads = 384;
constexpr int kRegsSoftmax = 216;
constexpr int kRegsProducer = 72;
static_assert(256 * kRegsSoftmax + 128 * kRegsProducer <= kThreads * 168, "register split");

constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Failure sites recorded in DeviceStatus::where.
enum Site : int {
  kSiteHeader = 1,
  kSiteLoadQEmpty = 10,
  kSiteLoadKvEmpty = 11,
  kSiteLoadOstFull = 12,
  kSiteMmaQFull = 20,
  kSiteMmaKvFull = 21,
  kSiteMmaPFull = 22,
  kSiteMmaOEmpty = 23,
  kSiteMmaDrain = 24,
  kSiteMmaTurn = 25,
  kSiteMmaDebugStall = 26,
  kSiteSmxSFull = 30,
  kSiteSmxOFull = 31,
  kSiteSmxOstEmpty = 34,
};

// PAIR: the CTA is one of a pair (a cluster of two) whose MMAs span both
// CTAs (M = 256, cta_group::2).  Each CTA then stages its own Q tiles and
// half of every key / value tile: keys [64 r, 64 r + 64) of a K tile and
// columns [64 r, 64 r + 64) of a V tile for the CTA of rank r, 16 KB either
// way, so a ring stage holds 16 KB instead of a whole 32 KB tile.
// OST: the epilogue stages each O tile in shared memory for a TMA store.
template <int D, bool PAIR = false, bool OST = false>
struct Cfg {
  static_assert(!PAIR || D == 128, "the CTA-pair forward is built for D = 128");
  static_assert(!(PAIR && OST), "the staged O store is a one-CTA form");
  static constexpr int kHalfBytes = kTileM * 64 * 2;  // 128 rows x 64 bf16, 128-byte swizzle
  static constexpr int kHalves = D / 64;
  static constexpr int kTileBytes = kHalves * kHalfBytes;
  static constexpr int kKPartHalfBytes = 64 * 64 * 2;  // PAIR: 64 keys x 64 columns of K
  static_assert(kKPartHalfBytes % 1024 == 0, "half-tile alignment");
  static constexpr int kStageBytes = PAIR ? kTileBytes / 2 : kTileBytes;
  // K/V ring: at D = 128 five 32 KB stages where the shared memory allows
  // (causal GQA +1.1%, dense unchanged), four beside the O staging buffer
  static constexpr int kStages = PAIR ? 8 : ((D == 128) ? (OST ? 4 : 5) : 8);
  static constexpr int kOCol = 256;  // O_t at column 256 + t * D; S_t at t * 128
  static constexpr int kSmemQ = 0;
  static constexpr int kSmemKV = kSmemQ + 2 * kTileBytes;
  // O staging for the epilogue's TMA store (one tile, OST only)
  static constexpr int kSmemOst = kSmemKV + kStages * kStageBytes;
  static constexpr int kSmemBar = kSmemOst + (OST ? kTileBytes : 0);
  // barriers: q_full[2] q_empty[2] kv_full[S] kv_empty[S] s_full[2] p_full[2]
  //           o_full[2] o_empty[2] drain never (the test hook's); OST:
  //           staged_full staged_empty
  static constexpr int kNumBars =
      2 + 2 + kStages + kStages + 2 + 2 + 2 + 2 + 1 + 1 + (OST ? 2 : 0);
  static constexpr int kSmemMisc = kSmemBar + 8 * kNumBars;
  static constexpr int kSmemDoc = (kSmemMisc + 16 + 15) / 16 * 16;  // int sdoc[2][128]
  static constexpr int kSmemBytes = kSmemDoc + 2 * kTileN * 4;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;  // slack for 1024-byte alignment
  static_assert(kSmemAlloc <= 227 * 1024, "shared memory per CTA");
};


struct KParams {
  CUtensorMap tmap_q;
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  CUtensorMap tmap_kh;  // K with 64-row boxes (the CTA pair's half tiles)
  __nv_bfloat16* out;
  float* lse;
  int B, H, H_kv, S_q, S_k, group;
  float scale;
  float scale_log2;  // scale * log2(e)
  uint32_t mask_flags;
  int window, q_offset;
  const int32_t* doc_ids;
  const int32_t* prefix_len;
  const float* alibi_slopes;
  int alibi_on;           // the BIAS variant also serves a bias table alone
  const float* rel_bias;  // [H][2 rel_max + 1], or null
  int rel_max;
  const uint8_t* blocks;  // user block map the mask was built from (header check)
  float softcap;
  const BlockMaskHeader* hdr;
  const int32_t* order;
  const int32_t* cnt;
  const uint32_t* list;
  const int32_t* doc_lo;  // [bm][S_k] first key of each token's document
  const int32_t* doc_hi;  // [bm][S_k] last key
  int nK, nP, bm, n_entries, n_items;
  int force_partial;
  DeviceStatus* status;
  float tau;
  uint64_t budget_ns;
  int poly_chunks;  // 16-column chunks per row (of 8) whose exp2 uses the polynomial
  int debug_stall;  // test hook (see ATTN_OPT_DEBUG_STALL)
  // soft cap on the FMA pipes: t = v Q(v^2) with Q's coefficients tq (the
  // fit of tanh_poly.h scaled by cap log2(e) and powers of u / v) while
  // |v| <= tlim; else y = v ty and the exp2 / reciprocal formula
  float tq[3];
  float tlim;
  float ty;
  CUtensorMap tmap_o;  // O, for the staged epilogue's TMA store
};

struct Ctl {
  volatile int* abort;   // generic pointer, for stores
  uint32_t abort_smem;   // the same flag's shared-memory address, for polling
  DeviceStatus* status;
  uint64_t budget_ns;
};

// Records the first failure and raises the abort flag (PAIR: of both CTAs).
template <bool PAIR>
__device__ __noinline__ void report(const Ctl& c, int code, int site, int detail) {
  if (atomicCAS(&c.status->code, 0, code) == 0) {
    c.status->where = site;
    c.status->block = blockIdx.x;
    c.status->detail = detail;
  }
  *c.abort = 1;
  if constexpr (PAIR) ptx::st_cluster_u32(ptx::mapa(c.abort_smem, ptx::cluster_ctarank() ^ 1u), 1u);
}

// Bounded wait on an mbarrier phase.  Returns false when the wait was given
// up (timeout here, or another role already aborted).  A waiting warp shares
// its SM sub-partition with a softmax warp that is working, so the wait
// sleeps in hardware (try_wait with a suspend hint, resumed as soon as the
// phase completes) and checks the abort flag and the time budget only every
// 16 suspensions, instead of spinning through the issue slots.
constexpr uint32_t kSuspendHintNs = 20000;
// After an abort, how long rank 1 of a CTA pair lets its copies in flight
// land before it leaves (they complete on rank 0's barriers, which it cannot
// poll): far above the latency of one tile copy.
constexpr uint64_t kPeerDrainNs = 200000;
// Phases completed by the peer CTA of a pair need no cluster-scope acquire
// either: the data behind every such barrier is Tensor Memory or shared
// memory filled by TMA, whose visibility the tcgen05 fences and the
// transaction count give.
template <bool PAIR>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& c, int site) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = 0;
  for (uint32_t spin = 1;; ++spin) {
    if (ptx::mbar_try_wait_hint(bar, parity, kSuspendHintNs)) return true;
    if ((spin & 15) == 0) {
      if (ptx::ld_volatile_shared(c.abort_smem)) return false;
      const uint64_t now = ptx::globaltimer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > c.budget_ns) {
        report<PAIR>(c, ATTN_ERR_TIMEOUT, site, (int)parity);
        return false;
      }
    }
  }
}

// Item w -> (batch, head, entry, half).  Entries are (mask batch, group of
// query tiles) ordered by descending work; when every entry has the same
// work the entries of one (batch, head) run next to each other so their K/V
// stay in L2.  A single CTA takes two query tiles at a time, so an entry of
// four tiles gives it two items, half 0 and 1 (HALVES).
struct Item {
  int b, h, e, pair, half;
};
template <bool HALVES>
__device__ __forceinline__ Item decode_item(const KParams& p, int w, int uniform) {
  Item it;
  it.half = 0;
  if constexpr (HALVES) {
    it.half = w & 1;
    w >>= 1;
  }
  const int nb = p.B / p.bm;  // batches sharing one mask entry
  int b_local;
  if (uniform) {
    it.e = w % p.n_entries;
    int rest = w / p.n_entries;
    b_local = rest / p.H;
    it.h = rest % p.H;
  } else {
    const int nbh = nb * p.H;
    int r = w / nbh;
    int rem = w % nbh;
    it.e = p.order[r];
    b_local = rem / p.H;
    it.h = rem % p.H;
  }
  const int bb = it.e / p.nP;
  it.pair = it.e % p.nP;
  it.b = (p.bm == 1) ? b_local : bb;
  return it;
}

// Static snake schedule over the items: round r gives unit c (a CTA, or a
// CTA pair) of G item r*G + c (even r) or r*G + G-1-c (odd r).
template <bool PAIR>
__device__ __forceinline__ int item_of(int r) {
  const int G = PAIR ? (int)ptx::cluster_count_x() : (int)gridDim.x;
  const int c = PAIR ? (int)ptx::cluster_id_x() : (int)blockIdx.x;
  return r * G + ((r & 1) ? (G - 1 - c) : c);
}
// Rounds of the snake schedule that hold an item for this CTA (or pair).
template <bool PAIR>
__device__ __forceinline__ int rounds_of(int n_items) {
  const int G = PAIR ? (int)ptx::cluster_count_x() : (int)gridDim.x;
  const int full = n_items / G;
  return full + (item_of<PAIR>(full) < n_items ? 1 : 0);
}

// Descriptor bits that do not depend on the start address: K-major tiles
// (Q, K) and the MN-major V tile.  A full descriptor is this constant plus
// (smem address >> 4); all addresses are below 256 KB, so the 14-bit start
// field never carries into the other fields.
template <int D>
struct Desc {
  static constexpr uint64_t kKMajor = ptx::smem_desc_sw128(0, 16, 1024);
  static constexpr uint64_t kVMajor = ptx::smem_desc_sw128(0, Cfg<D>::kHalfBytes, 1024);
};

// S = Q K^T: D/16 MMAs (K = 16 each) over the two 64-column halves of the
// swizzled tiles.  Warp-wide; one elected lane issues.  PAIR: M = 256 rows
// over the CTA pair, each CTA's K part 64 keys deep (8 KB per column half).
template <int D, bool PAIR>
__device__ __forceinline__ void issue_s(uint32_t tmem_s, uint64_t q_desc, uint64_t k_desc) {
  constexpr uint32_t idesc = ptx::idesc_bf16_f32(PAIR ? 2 * kTileM : kTileM, kTileN, false);
  constexpr int kKHalf = PAIR ? Cfg<D, PAIR>::kKPartHalfBytes : Cfg<D, PAIR>::kHalfBytes;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t qoff = (uint64_t)(((kk / 4) * Cfg<D, PAIR>::kHalfBytes + (kk % 4) * 32) >> 4);
    const uint64_t koff = (uint64_t)(((kk / 4) * kKHalf + (kk % 4) * 32) >> 4);
    if constexpr (PAIR)
      ptx::mma_ss_pair_elect(tmem_s, q_desc + qoff, k_desc + koff, idesc, kk > 0 ? 1u : 0u);
    else
      ptx::mma_ss_elect(tmem_s, q_desc + qoff, k_desc + koff, idesc, kk > 0 ? 1u : 0u);
  }
}

// O (+)= P V: 8 MMAs of 16 keys (16 rows of V = 2 KB of the swizzled tile;
// 8 packed bf16 columns of P in Tensor Memory).  Warp-wide.  PAIR: M = 256,
// each CTA's V part is its 64 columns of the tile.
template <int D, bool PAIR>
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint64_t v_desc,
                                         bool accumulate) {
  constexpr uint32_t idesc = ptx::idesc_bf16_f32(PAIR ? 2 * kTileM : kTileM, D, true);
#pragma unroll
  for (int kk = 0; kk < kTileN / 16; ++kk) {
    const uint32_t tp = tmem_p + (uint32_t)(kk * 8);
    const uint64_t vd = v_desc + (uint64_t)((kk * 2048) >> 4);
    const uint32_t acc = (accumulate || kk > 0) ? 1u : 0u;
    if constexpr (PAIR)
      ptx::mma_ts_pair_elect(tmem_o, tp, vd, idesc, acc);
    else
      ptx::mma_ts_elect(tmem_o, tp, vd, idesc, acc);
  }
}

// QUAD: the block mask groups four query tiles per entry (kTilesPerQuad);
// a CTA pair always uses such masks, a single CTA takes them in halves.
template <int D, bool ALIBI, bool SOFTCAP, bool PAIR, bool QUAD>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ KParams p) {
  static_assert(!PAIR || QUAD, "a CTA pair works on four-tile entries");
  // The one-CTA soft-cap and position-bias forms stage O in shared memory
  // and the Q loader warp stores it with TMA, so their softmax warps do not
  // wait at item boundaries while the O stores drain (with a sliding window
  // every CTA reaches them at about the same time; documents have short
  // items).  The plain form keeps direct stores: its items are long.
  constexpr bool kOst = (SOFTCAP || ALIBI) && !PAIR;
  using C = Cfg<D, PAIR, kOst>;
  constexpr int kTpe = QUAD ? kTilesPerQuad : kTilesPerItem;  // query tiles per entry
  constexpr bool kHalves = QUAD && !PAIR;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Launched with programmatic stream serialization: this CTA may start while
  // the kernel before it (normally the block-mask build) finishes, and reads
  // no global memory until that kernel's writes are visible.
  ptx::griddep_wait();

  // ---- block-mask consistency (uniform across the CTA) -------------------
  const BlockMaskHeader* hdr = p.hdr;
  const bool hdr_ok = hdr->magic == kBlockMaskMagic && hdr->version == kBlockMaskVersion &&
                      hdr->B == p.B && hdr->S_q == p.S_q && hdr->S_k == p.S_k &&
                      hdr->mask_flags == p.mask_flags && hdr->nP == p.nP && hdr->bm == p.bm &&
                      hdr->nK == p.nK &&
                      (!(p.mask_flags & ATTN_MASK_WINDOW) || hdr->window == p.window) &&
                      hdr->q_offset == p.q_offset &&
                      hdr->doc_ptr == reinterpret_cast<uint64_t>(p.doc_ids) &&
                      hdr->prefix_ptr == reinterpret_cast<uint64_t>(p.prefix_len) &&
                      hdr->blocks_ptr == reinterpret_cast<uint64_t>(p.blocks) &&
                      hdr->tiles_per_entry == kTpe;
  if (!hdr_ok) {
    if (threadIdx.x == 0 && atomicCAS(&p.status->code, 0, ATTN_ERR_DEVICE_CHECK) == 0) {
      p.status->where = kSiteHeader;
      p.status->block = blockIdx.x;
      p.status->detail = 0;
    }
    return;
  }
  const int uniform = hdr->uniform;
  const int docs_sorted = hdr->docs_sorted;
  // The r-th item of this CTA.  The soft-cap variant takes its items in
  // reverse when their work differs: with a sliding window nearly every item
  // has the same length, so in schedule order all CTAs reach their item
  // boundaries (and the O stores there) together; starting the CTAs whose
  // last item is short with that item staggers them (window 1024 + soft cap
  // +1.3%).  The other variants keep the schedule order: the same change cost
  // them 1-2% through the code of their item loop alone.
  int n_rev = 0;
  if constexpr (SOFTCAP) n_rev = uniform ? 0 : rounds_of<PAIR>(p.n_items);
  auto my_item = [&](int r) {
    if constexpr (SOFTCAP) {
      if (n_rev > 0) return r < n_rev ? item_of<PAIR>(n_rev - 1 - r) : p.n_items;
    }
    return item_of<PAIR>(r);
  };

  // ---- CTA pair --------------------------------------------------------
  // rank 0 issues every MMA of the pair; the work units of the persistent
  // schedule are CTA pairs.  Query tile t of this CTA within an item is
  // tile ci(t) of the block-mask entry.
  const int rank = PAIR ? (int)ptx::cluster_ctarank() : 0;
  auto ci = [&](const Item& it, int t) {
    return PAIR ? 2 * t + rank : (kHalves ? 2 * it.half + t : t);
  };

  // ---- shared memory map ------------------------------------------------
  auto bar = [&](int i) { return sbase + (uint32_t)(C::kSmemBar + 8 * i); };
  const int B_QF = 0, B_QE = 2, B_KVF = 4, B_KVE = 4 + C::kStages, B_SF = 4 + 2 * C::kStages,
            B_PF = B_SF + 2, B_OF = B_PF + 2, B_OE = B_OF + 2, B_DRAIN = B_OE + 2,
            B_NEVER = B_DRAIN + 1, B_OSTF = B_NEVER + 1, B_OSTE = B_NEVER + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::kSmemMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::kSmemMisc + 4);
  volatile int* s_turn = reinterpret_cast<volatile int*>(smem + C::kSmemMisc + 8);
  int* s_doc = reinterpret_cast<int*>(smem + C::kSmemDoc);

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(B_QF + 0), 1);
    ptx::mbar_init(bar(B_QF + 1), 1);
    ptx::mbar_init(bar(B_QE + 0), 1);
    ptx::mbar_init(bar(B_QE + 1), 1);
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(bar(B_KVF + s), 1);
      ptx::mbar_init(bar(B_KVE + s), 2);  // one commit per MMA issuer
    }
    for (int t = 0; t < 2; ++t) {
      // P ready / O free: one arrival per softmax warp (of both CTAs of a
      // pair, on rank 0's barriers)
      ptx::mbar_init(bar(B_SF + t), 1);
      ptx::mbar_init(bar(B_PF + t), PAIR ? 8 : 4);
      ptx::mbar_init(bar(B_OF + t), 1);
      ptx::mbar_init(bar(B_OE + t), PAIR ? 8 : 4);
    }
    ptx::mbar_init(bar(B_DRAIN), 2);
    ptx::mbar_init(bar(B_NEVER), 1);
    if constexpr (kOst) {
      ptx::mbar_init(bar(B_OSTF), 4);  // staged O tile full: one arrival per softmax warp
      ptx::mbar_init(bar(B_OSTE), 1);  // staged O tile read by its TMA store
    }
    *s_abort = 0;
    *s_turn = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    // a pair allocates the same columns in both CTAs, one warp of each
    if constexpr (PAIR) {
      ptx::tmem_alloc_pair(ptx::smem_addr(s_tmem), kTmemCols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(ptx::smem_addr(s_tmem), kTmemCols);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  // a pair's barriers must be initialised before the peer signals them
  if constexpr (PAIR)
    ptx::cluster_sync();
  else
    __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *s_tmem;

  Ctl ctl{s_abort, sbase + (uint32_t)(C::kSmemMisc + 4), p.status, p.budget_ns};
  const uint32_t s_turn_smem = sbase + (uint32_t)(C::kSmemMisc + 8);
  // rank 0's copy of barrier i (the pair's shared barriers live there)
  auto bar0 = [&](int i) { return PAIR ? ptx::mapa(bar(i), 0u) : bar(i); };

  if (warp >= 8) {
    // Producer warpgroup: give registers away first (whole warpgroup).
    ptx::setmaxnreg_dec<kRegsProducer>();
    if (warp == kLoadWarp && lane == 0) {
      // ===================== TMA producer: K / V ring ====================
      // Streams the key/value tiles of every item back to back, so the next
      // item's first tiles load while the current item finishes.
      // PAIR: each CTA loads its part of every tile (K: its 64 keys, V:
      // its 64 columns) and the copies of both CTAs complete on rank 0's
      // full barrier, which rank 0 arms for the bytes of both parts.
      ptx::prefetch_tmap(PAIR ? &p.tmap_kh : &p.tmap_k);
      ptx::prefetch_tmap(&p.tmap_v);
      const uint64_t pol_kv = ptx::policy_evict_last();
      uint32_t kv_cnt = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int w = my_item(r);
        if (w >= p.n_items) break;
        const Item it = decode_item<kHalves>(p, w, uniform);
        const int n = p.cnt[it.e];
        if (n == 0) continue;
        const uint32_t* lst = p.list + (size_t)it.e * p.nK;
        const int kvz = it.b * p.H_kv + it.h / p.group;
        for (int j = 0; j < n && ok; ++j) {
          const int row0 = (int)entry_tile(lst[j]) * kTileN;
          for (int which = 0; which < 2; ++which) {
            const int st = (int)(kv_cnt % C::kStages);
            if (kv_cnt >= (uint32_t)C::kStages) {
              ok = wait_bar<PAIR>(bar(B_KVE + st), ((kv_cnt / C::kStages) - 1) & 1, ctl,
                                  kSiteLoadKvEmpty);
              if (!ok) break;
            }
            const uint32_t dst = sbase + C::kSmemKV + st * C::kStageBytes;
            if constexpr (PAIR) {
              if (rank == 0) ptx::mbar_arrive_expect_tx(bar(B_KVF + st), 2 * C::kStageBytes);
              const uint32_t cb = bar0(B_KVF + st);
              if (which == 0) {
#pragma unroll
                for (int hx = 0; hx < C::kHalves; ++hx)
                  ptx::tma_load_3d_pair(dst + hx * C::kKPartHalfBytes, &p.tmap_kh, cb, hx * 64,
                                        row0 + 64 * rank, kvz, pol_kv);
              } else {
                ptx::tma_load_3d_pair(dst, &p.tmap_v, cb, 64 * rank, row0, kvz, pol_kv);
              }
            } else {
              ptx::mbar_arrive_expect_tx(bar(B_KVF + st), C::kTileBytes);
              const CUtensorMap* map = which == 0 ? &p.tmap_k : &p.tmap_v;
#pragma unroll
              for (int hx = 0; hx < C::kHalves; ++hx)
                ptx::tma_load_3d(dst + hx * C::kHalfBytes, map, bar(B_KVF + st), hx * 64, row0,
                                 kvz, pol_kv);
            }
            ++kv_cnt;
          }
        }
      }
      if (!ok) {
        // Let the copies already issued land before the CTA exits: wait (with
        // a bound) for the last phase issued on every stage still in use.
        // Rank 1 of a pair cannot see its copies complete (they count on
        // rank 0's barriers) and waits a fixed time instead.
        if (PAIR && rank != 0) {
          const uint64_t t0 = ptx::globaltimer_ns();
          while (ptx::globaltimer_ns() - t0 < kPeerDrainNs) {
          }
        } else {
          const uint32_t first = kv_cnt > (uint32_t)C::kStages ? kv_cnt - C::kStages : 0;
          for (uint32_t c = first; c < kv_cnt; ++c) {
            const uint64_t t0 = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(bar(B_KVF + (int)(c % C::kStages)), (c / C::kStages) & 1) &&
                   ptx::globaltimer_ns() - t0 < ctl.budget_ns) {
            }
          }
        }
      }
    } else if (warp == kQLoadWarp && lane == 0) {
      // ===================== TMA producer: Q tiles =======================
      // Loads Q_t of the next item as soon as the last S_t MMA of the
      // current item has read its buffer, independently of the K/V stream.
      // PAIR: each CTA loads its own query tiles; the copies complete on
      // rank 0's barrier, armed by rank 0 for both CTAs' bytes.
      ptx::prefetch_tmap(&p.tmap_q);
      if constexpr (kOst) ptx::prefetch_tmap(&p.tmap_o);
      const uint64_t pol_q = ptx::policy_evict_first();
      int act = 0;
      bool ok = true;
      int q_phase[2] = {-1, -1};  // parity of the last Q_t load issued
      // OST: this thread also stores the O tiles the softmax warpgroups stage
      // in shared memory, one item behind its Q loads (tile 0, then tile 1
      // of each item: the order in which the staging buffer is handed over).
      int prev_row0[2] = {0, 0}, prev_bh = 0;
      auto store_o = [&](int a) -> bool {
        for (int t = 0; t < 2; ++t) {
          const int e = 2 * a + t;
          if (!wait_bar<PAIR>(bar(B_OSTF), (uint32_t)(e & 1), ctl, kSiteLoadOstFull)) return false;
          if (prev_row0[t] < p.S_q) {  // a tile wholly past S_q has nothing to store
#pragma unroll
            for (int hx = 0; hx < C::kHalves; ++hx)
              ptx::tma_store_3d(&p.tmap_o, sbase + C::kSmemOst + hx * C::kHalfBytes, hx * 64,
                                prev_row0[t], prev_bh);
          }
          ptx::bulk_commit_group();
          ptx::bulk_wait_group_read0();
          ptx::mbar_arrive(bar(B_OSTE));
        }
        return true;
      };
      for (int r = 0; ok; ++r) {
        const int w = my_item(r);
        if (w >= p.n_items) break;
        const Item it = decode_item<kHalves>(p, w, uniform);
        if (p.cnt[it.e] == 0) continue;
        for (int t = 0; t < 2 && ok; ++t) {
          if (act > 0) ok = wait_bar<PAIR>(bar(B_QE + t), (act - 1) & 1, ctl, kSiteLoadQEmpty);
          if (!ok) break;
          const int row0 = (it.pair * kTpe + ci(it, t)) * kTileM;
          const uint32_t dst = sbase + C::kSmemQ + t * C::kTileBytes;
          if constexpr (PAIR) {
            if (rank == 0) ptx::mbar_arrive_expect_tx(bar(B_QF + t), 2 * C::kTileBytes);
            const uint32_t cb = bar0(B_QF + t);
#pragma unroll
            for (int hx = 0; hx < C::kHalves; ++hx)
              ptx::tma_load_3d_pair(dst + hx * C::kHalfBytes, &p.tmap_q, cb, hx * 64, row0,
                                    it.b * p.H + it.h, pol_q);
          } else {
            ptx::mbar_arrive_expect_tx(bar(B_QF + t), C::kTileBytes);
#pragma unroll
            for (int hx = 0; hx < C::kHalves; ++hx)
              ptx::tma_load_3d(dst + hx * C::kHalfBytes, &p.tmap_q, bar(B_QF + t), hx * 64, row0,
                               it.b * p.H + it.h, pol_q);
          }
          q_phase[t] = act & 1;
        }
        if constexpr (kOst) {
          if (ok && act > 0) ok = store_o(act - 1);
          for (int t = 0; t < 2; ++t) prev_row0[t] = (it.pair * kTpe + ci(it, t)) * kTileM;
          prev_bh = it.b * p.H + it.h;
        }
        ++act;
      }
      if constexpr (kOst) {
        if (ok && act > 0) ok = store_o(act - 1);
        ptx::bulk_wait_group0();  // every O store has landed before the CTA exits
      }
      if (!ok) {
        if (PAIR && rank != 0) {
          const uint64_t t0 = ptx::globaltimer_ns();
          while (ptx::globaltimer_ns() - t0 < kPeerDrainNs) {
          }
        } else {
          for (int t = 0; t < 2; ++t) {
            if (q_phase[t] < 0) continue;
            const uint64_t t0 = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(bar(B_QF + t), (uint32_t)q_phase[t]) &&
                   ptx::globaltimer_ns() - t0 < ctl.budget_ns) {
            }
          }
        }
      }
    } else if ((warp == kMmaWarp || warp == kMmaWarp + 1) && rank == 0) {
      // ===================== MMA issuers =================================
      // Two issuing warps, one per query tile.  tcgen05.mma issue blocks
      // until the tensor pipe accepts the MMA, and every mbarrier wait costs
      // a few hundred cycles even when the phase is already complete, so a
      // single issuer leaves the pipe idle during its waits; with one issuer
      // per tile the other tile's MMAs fill those gaps.  Each tile's chain
      //   S_t(0), PV_t(0), S_t(1), PV_t(1), ...
      // stays in issue order on one warp, which keeps the P_t / S_t aliasing
      // safe.  K/V stages are released once both issuers commit.  A turn
      // token makes the two tiles' MMA groups alternate on the pipe (tile 0
      // group k, tile 1 group k, tile 0 group k+1, ...) so each tile's S
      // finishes as early as in a strict ping-pong; an issuer does its
      // barrier waits while the other one issues, then takes its turn.
      // Every group waits only on earlier groups, so the order cannot
      // deadlock.  The loop is warp-uniform (all lanes wait and compute the
      // same descriptors, one elected lane issues), which keeps descriptors
      // in uniform registers and the MMAs back to back.
      //
      // PAIR: only rank 0 issues; each MMA spans both CTAs, and each commit
      // arrives on the barrier of that name in both CTAs (the peer's
      // softmax and producers wait on their own copies).
      const int t = warp - kMmaWarp;
      const uint32_t tS = tmem + (uint32_t)(t * kTileN);
      const uint32_t tO = tmem + (uint32_t)(C::kOCol + t * D);
      const uint64_t q_desc = Desc<D>::kKMajor + ((sbase + C::kSmemQ + t * C::kTileBytes) >> 4);
      const uint64_t kv0 = (sbase + C::kSmemKV) >> 4;
      auto stage = [&](uint32_t idx) { return idx % C::kStages; };
      auto k_desc = [&](uint32_t idx) {
        return Desc<D>::kKMajor + kv0 + (uint64_t)(stage(idx) * (C::kStageBytes >> 4));
      };
      auto v_desc = [&](uint32_t idx) {
        return Desc<D>::kVMajor + kv0 + (uint64_t)(stage(idx) * (C::kStageBytes >> 4));
      };
      auto kv_full = [&](uint32_t idx) { return bar(B_KVF + (int)stage(idx)); };
      auto kv_empty = [&](uint32_t idx) { return bar(B_KVE + (int)stage(idx)); };
      auto kv_par = [&](uint32_t idx) { return (idx / C::kStages) & 1; };
      auto wait_all = [&](uint32_t b, uint32_t par, int site) {
        return __all_sync(0xffffffffu, wait_bar<PAIR>(b, par, ctl, site));
      };
      auto commit = [&](uint32_t b) {
        if constexpr (PAIR)
          ptx::mma_commit_pair_elect(b, (uint16_t)0x3);
        else
          ptx::mma_commit_elect(b);
      };
      int grp = 0;  // groups this issuer has issued
      auto take_turn = [&]() -> bool {
        const int want = 2 * grp + t;
        bool got = true;
        if (ptx::ld_volatile_shared(s_turn_smem) != want) {
          const uint64_t t0 = ptx::globaltimer_ns();
          for (uint32_t spin = 1;; ++spin) {
            if (ptx::ld_volatile_shared(s_turn_smem) == want) break;
            // back off: a tight poll steals issue slots from the two softmax
            // warps that share this SM sub-partition
            __nanosleep(32);
            if ((spin & 255) == 0) {
              if (ptx::ld_volatile_shared(ctl.abort_smem)) { got = false; break; }
              if (ptx::globaltimer_ns() - t0 > p.budget_ns) {
                if (lane == 0) report<PAIR>(ctl, ATTN_ERR_TIMEOUT, kSiteMmaTurn, want);
                got = false;
                break;
              }
            }
          }
        }
        return __all_sync(0xffffffffu, got);
      };
      auto pass_turn = [&]() {
        __syncwarp();
        if (lane == 0) *s_turn = 2 * grp + t + 1;
        ++grp;
      };
      uint32_t kv_cnt = 0;
      uint32_t p_cnt = 0;
      int act = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int w = my_item(r);
        if (w >= p.n_items) break;
        const Item it = decode_item<kHalves>(p, w, uniform);
        const int n = p.cnt[it.e];
        if (n == 0) continue;
        const uint32_t k0 = kv_cnt;
        if (p.debug_stall) {  // test hook: a wait nothing ever completes
          ok = wait_all(bar(B_NEVER), 0, kSiteMmaDebugStall);
          if (!ok) break;
        }
        ok = wait_all(bar(B_QF + t), act & 1, kSiteMmaQFull) &&
             wait_all(kv_full(k0), kv_par(k0), kSiteMmaKvFull) && take_turn();
        if (!ok) break;
        ptx::tc_fence_after();
        issue_s<D, PAIR>(tS, q_desc, k_desc(k0));
        pass_turn();
        commit(bar(B_SF + t));
        if (n == 1) commit(bar(B_QE + t));
        commit(kv_empty(k0));
        for (int j = 0; j < n && ok; ++j) {
          const uint32_t vi = k0 + 2 * j + 1;  // V_j
          const uint32_t ki = k0 + 2 * j + 2;  // K_{j+1}
          const bool has_next = j + 1 < n;
          // Each mbarrier check costs a few hundred cycles even when the phase
          // has long completed, so the checks that are normally satisfied
          // early (K/V landed, O free) come first and P -- normally the last
          // to arrive -- comes last, right before the turn.
          ok = wait_all(kv_full(vi), kv_par(vi), kSiteMmaKvFull);
          if (ok && has_next) ok = wait_all(kv_full(ki), kv_par(ki), kSiteMmaKvFull);
          if (ok && j == 0 && act > 0) ok = wait_all(bar(B_OE + t), (act - 1) & 1, kSiteMmaOEmpty);
          if (ok) ok = wait_all(bar(B_PF + t), p_cnt & 1, kSiteMmaPFull);
          if (ok) ok = take_turn();
          if (!ok) break;
          ++p_cnt;
          ptx::tc_fence_after();
          issue_pv<D, PAIR>(tO, tS, v_desc(vi), j > 0);
          if (has_next) issue_s<D, PAIR>(tS, q_desc, k_desc(ki));
          pass_turn();
          commit(kv_empty(vi));
          if (has_next) {
            commit(bar(B_SF + t));
            if (j + 2 == n) commit(bar(B_QE + t));
            commit(kv_empty(ki));
          } else {
            commit(bar(B_OF + t));
          }
        }
        kv_cnt = k0 + 2 * (uint32_t)n;
        ++act;
      }
      // Wait for every MMA of both issuers before Tensor Memory is freed.
      __syncwarp();
      if constexpr (PAIR)
        ptx::mma_commit_pair_elect(bar(B_DRAIN), (uint16_t)0x1);  // rank 0's barrier only
      else
        ptx::mma_commit_elect(bar(B_DRAIN));
      const uint64_t t0 = ptx::globaltimer_ns();
      bool drained = true;
      while (!ptx::mbar_try_wait(bar(B_DRAIN), 0)) {
        if (ptx::globaltimer_ns() - t0 > p.budget_ns) {
          drained = false;
          break;
        }
      }
      if (!__all_sync(0xffffffffu, drained) && lane == 0)
        report<PAIR>(ctl, ATTN_ERR_TIMEOUT, kSiteMmaDrain, 0);
    }
  } else {
    ptx::setmaxnreg_inc<kRegsSoftmax>();
    // ===================== softmax warpgroups ============================
    const int t = warp >> 2;          // query tile of this warpgroup
    const int wq = warp & 3;          // lane quarter of Tensor Memory
    const int row = wq * 32 + lane;   // row within the query tile
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t tS = lane_base + (uint32_t)(t * kTileN);
    const uint32_t tO = lane_base + (uint32_t)(C::kOCol + t * D);
    int* sdoc = s_doc + t * kTileN;
    const float tau = p.tau;
    // P ready / O free: arrivals on rank 0's barriers in a CTA pair
    auto arrive = [&](int i) {
      if constexpr (PAIR)
        ptx::mbar_arrive_cluster(bar0(i));
      else
        ptx::mbar_arrive(bar(i));
    };
    uint32_t s_cnt = 0;
    int act = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int w = my_item(r);
      if (w >= p.n_items) break;
      const Item it = decode_item<kHalves>(p, w, uniform);
      const int n = p.cnt[it.e];
      const int tc = ci(it, t);                             // tile of the entry
      const int i = (it.pair * kTpe + tc) * kTileM + row;  // query row
      const bool valid = i < p.S_q;
      const size_t row_id = ((size_t)it.b * p.H + it.h) * (size_t)p.S_q + (size_t)i;
      __nv_bfloat16* orow = p.out + row_id * D;
      if (n == 0) {
        if (valid) {
          uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
          if (p.lse) p.lse[row_id] = -INFINITY;
        }
        continue;
      }
      const uint32_t* lst = p.list + (size_t)it.e * p.nK;

      // Row constants.
      const int qpos = i + p.q_offset;
      int lo = 0, hi = p.S_k - 1;
      if (p.mask_flags & ATTN_MASK_CAUSAL) hi = min(hi, qpos);
      if (p.mask_flags & ATTN_MASK_WINDOW) {
        lo = max(lo, qpos - p.window + 1);
        hi = min(hi, qpos);
      }
      if (p.mask_flags & ATTN_MASK_PREFIX_LM) hi = min(hi, max(qpos, p.prefix_len[it.b] - 1));
      // Documents: with packed (non-decreasing) ids the keys of row i's
      // document form the interval [doc_lo[i], doc_hi[i]], folded into the
      // row's bounds; other ids are compared element by element.
      const bool has_doc = (p.mask_flags & ATTN_MASK_DOCUMENT) != 0 && !docs_sorted;
      if ((p.mask_flags & ATTN_MASK_DOCUMENT) && docs_sorted && valid) {
        const size_t di = (size_t)it.b * p.S_k + (size_t)i;
        lo = max(lo, p.doc_lo[di]);
        hi = min(hi, p.doc_hi[di]);
      }
      const int* doc_b = has_doc ? p.doc_ids + (size_t)it.b * p.S_k : nullptr;
      const int doc_i = (has_doc && valid) ? doc_b[i] : 0;
      float slope2 = 0.f;  // ALiBi slope in the units of the transformed score
      if constexpr (ALIBI) {
        if (p.alibi_on) {
          float m = p.alibi_slopes ? p.alibi_slopes[it.h]
                                   : exp2f(-8.0f * (float)(it.h + 1) / (float)p.H);
          slope2 = SOFTCAP ? m * (2.0f * kLog2e / p.softcap) : m * kLog2e;
        }
      }
      // relative-position bias table row of this head, and its factor to
      // the units of the transformed score
      const float* relrow =
          p.rel_bias ? p.rel_bias + (size_t)it.h * (2 * (size_t)p.rel_max + 1) : nullptr;
      const float rel_scale = SOFTCAP ? 2.0f * kLog2e / p.softcap : kLog2e;
      // Score transform coefficients.
      //   plain:   t = s * scale * log2(e)             (folded into the exp)
      //   ALiBi:   t = s * scale * log2(e) + slope2 * (j - qpos)
      //   softcap: y = (s * scale + bias) * 2 log2(e) / cap,
      //            t = cap log2(e) * (1 - 2 / (2^y + 1))
      const float sc = SOFTCAP ? p.scale * (2.0f * kLog2e / p.softcap) : p.scale_log2;
      const float capl2 = p.softcap * kLog2e;

      float m_ref = -INFINITY;  // reference max, log2 units
      float l = 0.f;            // running sum of 2^(t - m_ref)

      for (int j = 0; j < n && ok; ++j) {
        const uint32_t entry = lst[j];
        const int kt = (int)entry_tile(entry);
        const uint32_t cls = entry_cls(entry, tc);
        const int j0 = kt * kTileN;
        bool got = wait_bar<PAIR>(bar(B_SF + t), s_cnt & 1, ctl, kSiteSmxSFull);
        ok = __all_sync(0xffffffffu, got);
        if (!ok) break;
        ++s_cnt;
        ptx::tc_fence_after();
        // Doc ids of this key tile into shared memory (whole warpgroup).  S_t(j)
        // is issued only after all four warps released P_t(j-1), so no warp is
        // still reading the previous tile's ids.
        if (has_doc && cls == kPartial) {
          const int jj = j0 + row;
          sdoc[row] = (jj < p.S_k) ? doc_b[jj] : INT32_MIN;
          ptx::named_bar_sync(1 + t, 128);
        }

        if (cls == kEmpty) {
          uint32_t z[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) z[c] = 0u;
          ptx::tmem_st32(tS, z);
          ptx::tmem_st32(tS + 32u, z);
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive(B_PF + t);
        } else {
          float tv[kTileN];
          {
            // all four loads in flight before one wait
            uint32_t r0[32], r1[32], r2[32], r3[32];
            ptx::tmem_ld32(tS + 0u, r0);
            ptx::tmem_ld32(tS + 32u, r1);
            ptx::tmem_ld32(tS + 64u, r2);
            ptx::tmem_ld32(tS + 96u, r3);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              tv[c] = __uint_as_float(r0[c]);
              tv[32 + c] = __uint_as_float(r1[c]);
              tv[64 + c] = __uint_as_float(r2[c]);
              tv[96 + c] = __uint_as_float(r3[c]);
            }
          }
          if constexpr (SOFTCAP) {
            // score mods
            // relative-position bias: where the whole tile lies beyond +-R of
            // every row of the warp, the clamped bias is one table entry,
            // folded into the constant term below; otherwise a loop of its own
            // (a uniform branch, so the loops stay branch-free), scaled so it
            // adds table * rel_scale to s * sc
            float rel_const = 0.f;
            if constexpr (ALIBI) {
              if (relrow != nullptr) {
                const int lo_r = j0 - qpos, hi_r = j0 + kTileN - 1 - qpos;
                if (__all_sync(0xffffffffu, hi_r <= -p.rel_max)) {
                  rel_const = __ldg(relrow) * rel_scale;
                } else if (__all_sync(0xffffffffu, lo_r >= p.rel_max)) {
                  rel_const = __ldg(relrow + 2 * p.rel_max) * rel_scale;
                } else {
                  const float rs = rel_scale / sc;
#pragma unroll
                  for (int c = 0; c < kTileN; ++c) {
                    const int r = min(max(j0 + c - qpos, -p.rel_max), p.rel_max);
                    tv[c] = fmaf(__ldg(relrow + r + p.rel_max), rs, tv[c]);
                  }
                }
              }
              // additive position biases, paired fp32 instructions: the
              // exponent's log2 units, or with the soft cap the units of
              // y = 2 log2(e) x / cap, the cap itself following below
              const float b0 = fmaf(slope2, (float)(j0 - qpos), rel_const);
              const uint64_t sc2 = ptx::f2(sc, sc), sl2 = ptx::f2(slope2, slope2),
                             b02 = ptx::f2(b0, b0);
#pragma unroll
              for (int c = 0; c < kTileN; c += 2) {
                const uint64_t bias2 = ptx::ffma2(sl2, ptx::f2((float)c, (float)(c + 1)), b02);
                ptx::f2_split(ptx::ffma2(ptx::f2(tv[c], tv[c + 1]), sc2, bias2), tv[c], tv[c + 1]);
              }
            }
            // conditional rescale: the row's reference max moves only when the
            // tile's max exceeds it by more than tau; returns the max to
            // subtract in the exponent
            auto update_max = [&](float mx) -> float {
              const float m_new = fmaxf(m_ref, mx);
              const bool need = m_new > m_ref + tau;
              const bool had = m_ref != -INFINITY;
              float factor = 1.0f;
              if (need) {
                factor = ptx::ex2_approx(m_ref - m_new);
                l *= factor;
                m_ref = m_new;
              }
              const bool resc = need && had;
              if (__any_sync(0xffffffffu, resc)) {
                const float f = resc ? factor : 1.0f;
#pragma unroll
                for (int c4 = 0; c4 < D / 32; ++c4) {
                  uint32_t o[32];
                  ptx::tmem_ld32(tO + (uint32_t)(c4 * 32), o);
                  ptx::tmem_wait_ld();
#pragma unroll
                  for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * f);
                  ptx::tmem_st32(tO + (uint32_t)(c4 * 32), o);
                }
              }
              return (m_ref == -INFINITY) ? 0.f : m_ref;
            };
            float la[4] = {0.f, 0.f, 0.f, 0.f};
            // Soft cap t = cap log2(e) tanh(u) of the pre-cap value v (the raw
            // score, or y with position biases; u = kk v).  tanh is monotone,
            // so the row max is taken on v and capped once.  Where every
            // visible v of the warp's rows lies within |u| <= U0 -- always,
            // for scores of ordinary size -- tanh comes from the odd
            // polynomial of tanh_poly.h on the FMA pipes (pre-scaled:
            // t = v Q(v^2)); other tiles take t = C (1 - 2 / (2^y + 1)) on the
            // exp2 and reciprocal units ("FlashAttention-4 explained",
            // "Forward pass fixes": moving transcendental work off the MUFU
            // unit, whose reciprocal runs at half the exp2 rate on GB300).
            // On a PARTIAL tile the hidden v of a mixed chunk become NaN,
            // which the min / max instructions skip, so the range and the max
            // cover the visible scores only; their exponent argument is NaN
            // too and becomes -inf through fmaxf(NaN, -inf) = -inf, so their
            // exponential is exactly 0.  The two tile classes run separate
            // straight-line copies of this body.
            auto softcap_tile = [&](auto partial_tag) {
              constexpr bool kPart = decltype(partial_tag)::value;
              // On a PARTIAL tile each 32-column chunk is classified for the
              // warp's 32 rows: hidden for every row (bit k of hid; skipped by
              // the range, the max and the exponentials, its P stored as 0),
              // mixed (bit k of mix; hidden scores set to NaN one by one), or
              // visible for every row.  With a window or causal band, a
              // warp's rows differ by at most 31 positions, so on a diagonal
              // or window-edge tile one chunk is mixed and the others are
              // whole.  Document ids compared key by key make every chunk
              // that is not hidden mixed.
              uint32_t hid = 0u, mix = 0u;
              if constexpr (kPart) {
                const int clo = lo - j0, chi = hi - j0;
                const float qnan = __int_as_float(0x7fc00000);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const bool h = (chi < 32 * k) || (clo > 32 * k + 31);
                  const bool v = !has_doc && clo <= 32 * k && chi >= 32 * k + 31;
                  const bool all_h = __all_sync(0xffffffffu, h);
                  const bool all_v = __all_sync(0xffffffffu, v);
                  hid |= (uint32_t)all_h << k;
                  mix |= (uint32_t)!(all_h || all_v) << k;
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  if ((mix >> k) & 1u) {
                    if (has_doc) {
#pragma unroll
                      for (int c = 32 * k; c < 32 * k + 32; ++c) {
                        const bool vis = (c >= clo) & (c <= chi) & (sdoc[c] == doc_i);
                        tv[c] = vis ? tv[c] : qnan;
                      }
                    } else {
#pragma unroll
                      for (int c = 32 * k; c < 32 * k + 32; ++c) {
                        const bool vis = (c >= clo) & (c <= chi);
                        tv[c] = vis ? tv[c] : qnan;
                      }
                    }
                  }
                }
              }
              // row max and min, three-input instructions over four chains
              float vmax, vmin;
              {
                float mxa[4], mna[4];
                if constexpr (kPart) {
                  // chains start at NaN, which the min / max instructions skip
#pragma unroll
                  for (int a = 0; a < 4; ++a) mxa[a] = mna[a] = __int_as_float(0x7fc00000);
#pragma unroll
                  for (int k = 0; k < 4; ++k) {
                    if (!((hid >> k) & 1u)) {
#pragma unroll
                      for (int c = 32 * k; c < 32 * k + 32; c += 8) {
#pragma unroll
                        for (int a = 0; a < 4; ++a) {
                          mxa[a] = ptx::fmax3(mxa[a], tv[c + 2 * a], tv[c + 2 * a + 1]);
                          mna[a] = ptx::fmin3(mna[a], tv[c + 2 * a], tv[c + 2 * a + 1]);
                        }
                      }
                    }
                  }
                } else {
#pragma unroll
                  for (int a = 0; a < 4; ++a) {
                    mxa[a] = ptx::fmax3(tv[2 * a], tv[2 * a + 1], tv[8 + 2 * a]);
                    mna[a] = ptx::fmin3(tv[2 * a], tv[2 * a + 1], tv[8 + 2 * a]);
                  }
#pragma unroll
                  for (int a = 0; a < 4; ++a) {  // columns 9, 11, 13, 15
                    mxa[a] = fmaxf(mxa[a], tv[9 + 2 * a]);
                    mna[a] = fminf(mna[a], tv[9 + 2 * a]);
                  }
#pragma unroll
                  for (int c = 16; c < kTileN; c += 8) {
#pragma unroll
                    for (int a = 0; a < 4; ++a) {
                      mxa[a] = ptx::fmax3(mxa[a], tv[c + 2 * a], tv[c + 2 * a + 1]);
                      mna[a] = ptx::fmin3(mna[a], tv[c + 2 * a], tv[c + 2 * a + 1]);
                    }
                  }
                }
                vmax = fmaxf(fmaxf(mxa[0], mxa[1]), fmaxf(mxa[2], mxa[3]));
                vmin = fminf(fminf(mna[0], mna[1]), fminf(mna[2], mna[3]));
              }
              // NaN comparisons are false: a row with no visible score in
              // the tile (vmax NaN or -inf) counts as in range
              const bool poly = __all_sync(0xffffffffu, !(vmax > p.tlim) && !(vmin < -p.tlim));
              float mx;
              if (!(vmax > -INFINITY)) {
                mx = -INFINITY;
              } else if (poly) {
                const float w = vmax * vmax;
                float q = fmaf(p.tq[2], w, p.tq[1]);
                q = fmaf(q, w, p.tq[0]);
                mx = vmax * q;
              } else {
                const float e = ptx::ex2_approx(vmax * p.ty);
                mx = fmaf(ptx::rcp_approx(e + 1.0f), -2.0f * capl2, capl2);
              }
              const float m_use = update_max(mx);
              uint64_t acc2[2] = {0ull, 0ull};
              // the exponentials of P, 32 bf16 pairs of columns per Tensor
              // Memory store; arg(a, b, ea, eb) gives the exponent arguments
              // of two columns.  The exponent argument of a hidden score
              // (NaN) becomes -inf, so its exponential is exactly 0.
              auto exp_pass = [&](auto arg) {
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                  uint32_t pk[32];
#pragma unroll
                  for (int hf = 0; hf < 2; ++hf) {
                    if (kPart && ((hid >> (2 * h2 + hf)) & 1u)) {
#pragma unroll
                      for (int c = 16 * hf; c < 16 * hf + 16; ++c) pk[c] = 0u;
                    } else {
#pragma unroll
                      for (int c = 16 * hf; c < 16 * hf + 16; ++c) {
                        float pa, pb;
                        arg(tv[h2 * 64 + 2 * c], tv[h2 * 64 + 2 * c + 1], pa, pb);
                        if constexpr (kPart) {
                          pa = fmaxf(pa, -INFINITY);
                          pb = fmaxf(pb, -INFINITY);
                        }
                        pa = ptx::ex2_approx(pa);
                        pb = ptx::ex2_approx(pb);
                        acc2[c & 1] = ptx::fadd2(acc2[c & 1], ptx::f2(pa, pb));
                        pk[c] = ptx::pack_bf16x2(pa, pb);
                      }
                    }
                  }
                  ptx::tmem_st32(tS + (uint32_t)(h2 * 32), pk);
                }
              };
              if (poly) {
                const uint64_t q2 = ptx::f2(p.tq[2], p.tq[2]), q1 = ptx::f2(p.tq[1], p.tq[1]),
                               q0 = ptx::f2(p.tq[0], p.tq[0]), nm2 = ptx::f2(-m_use, -m_use);
                exp_pass([&](float a, float b, float& ea, float& eb) {
                  const uint64_t v2 = ptx::f2(a, b);
                  const uint64_t w2 = ptx::fmul2(v2, v2);
                  uint64_t r2 = ptx::ffma2(w2, q2, q1);
                  r2 = ptx::ffma2(r2, w2, q0);
                  ptx::f2_split(ptx::ffma2(v2, r2, nm2), ea, eb);
                });
              } else {
                const uint64_t ty2 = ptx::f2(p.ty, p.ty), one2 = ptx::f2(1.0f, 1.0f),
                               m2c2 = ptx::f2(-2.0f * capl2, -2.0f * capl2),
                               cm2 = ptx::f2(capl2 - m_use, capl2 - m_use);
                exp_pass([&](float a, float b, float& ea, float& eb) {
                  float xa, xb;
                  ptx::f2_split(ptx::fmul2(ptx::f2(a, b), ty2), xa, xb);
                  xa = ptx::ex2_approx(xa);
                  xb = ptx::ex2_approx(xb);
                  float da, db;
                  ptx::f2_split(ptx::fadd2(ptx::f2(xa, xb), one2), da, db);
                  ptx::f2_split(ptx::ffma2(ptx::f2(ptx::rcp_approx(da), ptx::rcp_approx(db)), m2c2,
                                           cm2),
                                ea, eb);
                });
              }
              ptx::f2_split(acc2[0], la[0], la[1]);
              ptx::f2_split(acc2[1], la[2], la[3]);
            };
            if (cls == kPartial)
              softcap_tile(std::true_type{});
            else
              softcap_tile(std::false_type{});
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive(B_PF + t);
            l += (la[0] + la[1]) + (la[2] + la[3]);
          } else {
          // score mods
          // relative-position bias: where the whole tile lies beyond +-R of
          // every row of the warp, the clamped bias is one table entry,
          // folded into the constant term below; otherwise a loop of its own
          // (a uniform branch, so the loops stay branch-free), scaled so it
          // adds table * rel_scale to s * sc
          float rel_const = 0.f;
          if constexpr (ALIBI) {
            if (relrow != nullptr) {
              const int lo_r = j0 - qpos, hi_r = j0 + kTileN - 1 - qpos;
              if (__all_sync(0xffffffffu, hi_r <= -p.rel_max)) {
                rel_const = __ldg(relrow) * rel_scale;
              } else if (__all_sync(0xffffffffu, lo_r >= p.rel_max)) {
                rel_const = __ldg(relrow + 2 * p.rel_max) * rel_scale;
              } else {
                const float rs = rel_scale / sc;
#pragma unroll
                for (int c = 0; c < kTileN; ++c) {
                  const int r = min(max(j0 + c - qpos, -p.rel_max), p.rel_max);
                  tv[c] = fmaf(__ldg(relrow + r + p.rel_max), rs, tv[c]);
                }
              }
            }
          }
          if constexpr (ALIBI) {
            // paired fp32 instructions, two columns at a time
            const float b0 = fmaf(slope2, (float)(j0 - qpos), rel_const);
            const uint64_t sc2 = ptx::f2(sc, sc), sl2 = ptx::f2(slope2, slope2),
                           b02 = ptx::f2(b0, b0);
#pragma unroll
            for (int c = 0; c < kTileN; c += 2) {
              const uint64_t bias2 = ptx::ffma2(sl2, ptx::f2((float)c, (float)(c + 1)), b02);
              uint64_t x2 = ptx::ffma2(ptx::f2(tv[c], tv[c + 1]), sc2, bias2);
              ptx::f2_split(x2, tv[c], tv[c + 1]);
            }
          }
          // mask (partial tiles only).  The position-bias variant masks by
          // 32-column chunks: a chunk that every row of the warp sees whole
          // is left as it is, the others are masked score by score (documents
          // + ALiBi +3%; a third branch that set a hidden chunk to -inf as a
          // whole made the kernel spill).  The plain variant, whose partial
          // tiles are few (the causal diagonal), keeps one loop: the chunked
          // form cost it 7% on dense and causal, where no tile is partial.
          if (cls == kPartial) {
            const int clo = lo - j0, chi = hi - j0;
            auto mask_cols = [&](int c0, int c1) {
              if (has_doc) {
#pragma unroll
                for (int c = c0; c < c1; ++c) {
                  const bool vis = (c >= clo) & (c <= chi) & (sdoc[c] == doc_i);
                  tv[c] = vis ? tv[c] : -INFINITY;
                }
              } else {
#pragma unroll
                for (int c = c0; c < c1; ++c) {
                  const bool vis = (c >= clo) & (c <= chi);
                  tv[c] = vis ? tv[c] : -INFINITY;
                }
              }
            };
            if constexpr (ALIBI) {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const bool all_v = __all_sync(0xffffffffu, !has_doc && clo <= 32 * k &&
                                                               chi >= 32 * k + 31);
                if (!all_v) mask_cols(32 * k, 32 * k + 32);
              }
            } else {
              mask_cols(0, kTileN);
            }
          }
          // row max: eight independent chains (measured faster on GB300 than
          // the three-input max)
          float mxa[8];
#pragma unroll
          for (int a = 0; a < 8; ++a) mxa[a] = tv[a];
#pragma unroll
          for (int c = 8; c < kTileN; c += 16) {
#pragma unroll
            for (int a = 0; a < 8; ++a) mxa[a] = fmaxf(fmaxf(mxa[a], tv[c + a]), tv[c + 8 + a]);
          }
          float mx = fmaxf(fmaxf(fmaxf(mxa[0], mxa[1]), fmaxf(mxa[2], mxa[3])),
                           fmaxf(fmaxf(mxa[4], mxa[5]), fmaxf(mxa[6], mxa[7])));
          constexpr bool kPlain = !ALIBI;
          const float xs = kPlain ? p.scale_log2 : 1.0f;  // raw scores still need the scale
          mx = kPlain ? mx * xs : mx;
          // conditional rescale
          const float m_new = fmaxf(m_ref, mx);
          const bool need = m_new > m_ref + tau;
          const bool had = m_ref != -INFINITY;
          float factor = 1.0f;
          if (need) {
            factor = ptx::ex2_approx(m_ref - m_new);
            l *= factor;
            m_ref = m_new;
          }
          const bool resc = need && had;
          if (__any_sync(0xffffffffu, resc)) {
            const float f = resc ? factor : 1.0f;
#pragma unroll
            for (int c4 = 0; c4 < D / 32; ++c4) {
              uint32_t o[32];
              ptx::tmem_ld32(tO + (uint32_t)(c4 * 32), o);
              ptx::tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * f);
              ptx::tmem_st32(tO + (uint32_t)(c4 * 32), o);
            }
          }
          const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
          // exponentials, row sum, bf16 P written over S.  The first
          // poly_chunks 16-column chunks of the row evaluate exp2 with the
          // FMA polynomial, the rest with the hardware unit ("FlashAttention-4
          // explained", "Forward pass fixes", "Software-emulated
          // exponentials"); the choice is uniform across the warp.
          float la[4] = {0.f, 0.f, 0.f, 0.f};
          const int npc = p.poly_chunks;
          if (npc == 0) {
            // hardware exp2 only: one straight-line loop (the chunked form
            // below schedules measurably worse).  The softmax is bound by
            // instruction issue, so the scale-and-subtract and the row sum use
            // paired fp32 instructions (two columns per instruction).
            const uint64_t xs2 = ptx::f2(xs, xs), nm2 = ptx::f2(-m_use, -m_use);
            uint64_t acc2[2] = {0ull, 0ull};
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              uint32_t pk[32];
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                float pa, pb;
                ptx::f2_split(ptx::ffma2(ptx::f2(tv[h2 * 64 + 2 * c], tv[h2 * 64 + 2 * c + 1]),
                                         xs2, nm2),
                              pa, pb);
                pa = ptx::ex2_approx(pa);
                pb = ptx::ex2_approx(pb);
                acc2[c & 1] = ptx::fadd2(acc2[c & 1], ptx::f2(pa, pb));
                pk[c] = ptx::pack_bf16x2(pa, pb);
              }
              ptx::tmem_st32(tS + (uint32_t)(h2 * 32), pk);
            }
            ptx::f2_split(acc2[0], la[0], la[1]);
            ptx::f2_split(acc2[1], la[2], la[3]);
          } else {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            uint32_t pk[32];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              if (h2 * 4 + q4 < npc) {
#pragma unroll
                for (int c = q4 * 8; c < q4 * 8 + 8; ++c) {
                  const float pa = ptx::exp2_poly(fmaf(tv[h2 * 64 + 2 * c], xs, -m_use));
                  const float pb = ptx::exp2_poly(fmaf(tv[h2 * 64 + 2 * c + 1], xs, -m_use));
                  la[(c & 1) * 2] += pa;
                  la[(c & 1) * 2 + 1] += pb;
                  pk[c] = ptx::pack_bf16x2(pa, pb);
                }
              } else {
#pragma unroll
                for (int c = q4 * 8; c < q4 * 8 + 8; ++c) {
                  const float pa = ptx::ex2_approx(fmaf(tv[h2 * 64 + 2 * c], xs, -m_use));
                  const float pb = ptx::ex2_approx(fmaf(tv[h2 * 64 + 2 * c + 1], xs, -m_use));
                  la[(c & 1) * 2] += pa;
                  la[(c & 1) * 2 + 1] += pb;
                  pk[c] = ptx::pack_bf16x2(pa, pb);
                }
              }
            }
            ptx::tmem_st32(tS + (uint32_t)(h2 * 32), pk);
          }
          }
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive(B_PF + t);
          l += (la[0] + la[1]) + (la[2] + la[3]);
          }
        }
      }
      if (!ok) break;

      // ---- epilogue: O / l -> bf16, LSE --------------------------------
      {
        bool got = wait_bar<PAIR>(bar(B_OF + t), act & 1, ctl, kSiteSmxOFull);
        ok = __all_sync(0xffffffffu, got);
        if (!ok) break;
      }
      ptx::tc_fence_after();
      // A row that never saw a visible key keeps m_ref = -inf: O = 0 and
      // LSE = -inf.
      const bool seen = m_ref != -INFINITY && l > 0.f;
      const float inv_l = seen ? 1.0f / l : 0.f;
      {
        // all of O's loads in flight before one wait; Tensor Memory is free
        // for the next item's first PV as soon as they have landed
        uint32_t o[D / 32][32];
#pragma unroll
        for (int c4 = 0; c4 < D / 32; ++c4) ptx::tmem_ld32(tO + (uint32_t)(c4 * 32), o[c4]);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive(B_OE + t);
        if constexpr (kOst) {
          // Stage the row for the Q loader's TMA store: 128-byte rows in each
          // 64-column half, 16-byte chunks swizzled by the row (the tensor
          // map's 128-byte swizzle), so the warp's stores spread over all
          // banks.  Rows past S_q are staged too; the store clips them.  The
          // buffer alternates between the tiles: epilogue e waits until
          // epilogue e - 1's store has read it.
          const int e = 2 * act + t;
          if (e > 0) {
            const bool got = wait_bar<PAIR>(bar(B_OSTE), (uint32_t)((e - 1) & 1), ctl,
                                            kSiteSmxOstEmpty);
            ok = __all_sync(0xffffffffu, got);
            if (!ok) break;
          }
          const uint32_t srow = sbase + C::kSmemOst + (uint32_t)(row * 128);
#pragma unroll
          for (int c4 = 0; c4 < D / 32; ++c4) {
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 16; ++c)
              pk[c] = ptx::pack_bf16x2(__uint_as_float(o[c4][2 * c]) * inv_l,
                                       __uint_as_float(o[c4][2 * c + 1]) * inv_l);
            const uint32_t half = srow + (uint32_t)((c4 / 2) * C::kHalfBytes);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              const int j = (c4 % 2) * 4 + cc;  // 16-byte chunk of the 128-byte row
              ptx::sts_v4(half + (uint32_t)((j ^ (row & 7)) * 16), pk[4 * cc], pk[4 * cc + 1],
                          pk[4 * cc + 2], pk[4 * cc + 3]);
            }
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(B_OSTF));
        } else {
        const bool out32 = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
        if (valid) {
#pragma unroll
          for (int c4 = 0; c4 < D / 32; ++c4) {
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 16; ++c)
              pk[c] = ptx::pack_bf16x2(__uint_as_float(o[c4][2 * c]) * inv_l,
                                       __uint_as_float(o[c4][2 * c + 1]) * inv_l);
            if (out32) {  // rows start 32-byte aligned: whole sectors per lane
              ptx::stg_v8(orow + c4 * 32, pk);
              ptx::stg_v8(orow + c4 * 32 + 16, pk + 8);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(orow + c4 * 32);
#pragma unroll
              for (int c = 0; c < 4; ++c)
                dst[c] = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            }
          }
        }
        }
      }
      if (valid && p.lse) p.lse[row_id] = seen ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
      ++act;
    }
  }

  // ---- teardown --------------------------------------------------------
  // A pair leaves together: rank 0's MMAs write the peer's Tensor Memory and
  // signal its barriers, and the peer's copies signal rank 0's, so neither
  // CTA frees or exits before both are done.
  ptx::tc_fence_before();
  if constexpr (PAIR)
    ptx::cluster_sync();
  else
    __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    ptx::tc_fence_after();
    if constexpr (PAIR)
      ptx::tmem_dealloc_pair(tmem, kTmemCols);
    else
      ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host ----

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// [rows_outer][S][D] bf16 viewed as 3-D (D, S, rows_outer); box 64 x
// box_rows x 1 with 128-byte swizzle.  Rows beyond S read as zero.
bool make_map(CUtensorMap* map, const void* ptr, int D, int S, int outer,
              int box_rows = kTileM) {
  EncodeTiledFn enc = get_encode_tiled();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)outer};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)S * (cuuint64_t)D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// grid: CTAs wanted (a CTA pair counts two); PAIR launches clusters of two
// and caps the grid at the pairs that fit on the GPU at once, so that every
// pair of the persistent schedule is resident.
// Launch-time queries that do not change for a device are made once per
// device and kernel instantiation: the opt-in shared memory size (a function
// attribute) and, for CTA pairs, how many clusters fit.  A concurrent first
// call only repeats the same idempotent query.
constexpr int kLaunchCacheDevices = 64;

template <int D, bool ALIBI, bool SOFTCAP, bool PAIR, bool QUAD>
cudaError_t launch_variant(const KParams& kp, int grid, cudaStream_t stream, int dev) {
  auto kern = attn_fwd_kernel<D, ALIBI, SOFTCAP, PAIR, QUAD>;
  static std::atomic<bool> attr_set[kLaunchCacheDevices];
  static std::atomic<int> clusters[kLaunchCacheDevices];
  const bool cache = dev >= 0 && dev < kLaunchCacheDevices;
  cudaError_t err = cudaSuccess;
  if (!cache || !attr_set[dev].load(std::memory_order_relaxed)) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Cfg<D, PAIR, (SOFTCAP || ALIBI) && !PAIR>::kSmemAlloc);
    if (err != cudaSuccess) return err;
    if (cache) attr_set[dev].store(true, std::memory_order_relaxed);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg<D, PAIR, (SOFTCAP || ALIBI) && !PAIR>::kSmemAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if constexpr (PAIR) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
    int pairs = (grid + 1) / 2;
    cfg.gridDim = dim3(2u * (unsigned)pairs, 1, 1);
    int resident = cache ? clusters[dev].load(std::memory_order_relaxed) : 0;
    if (resident == 0) {
      err = cudaOccupancyMaxActiveClusters(&resident, kern, &cfg);
      if (err != cudaSuccess) return err;
      if (resident < 1) return cudaErrorInvalidConfiguration;
      if (cache) clusters[dev].store(resident, std::memory_order_relaxed);
    }
    if (pairs > resident) pairs = resident;
    cfg.gridDim = dim3(2u * (unsigned)pairs, 1, 1);
  } else {
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
  }
  return cudaLaunchKernelEx(&cfg, kern, kp);
}

template <int D, bool PAIR, bool QUAD>
cudaError_t launch_d(const KParams& kp, bool alibi, bool softcap, int grid, cudaStream_t s,
                     int dev) {
  if (alibi && softcap) return launch_variant<D, true, true, PAIR, QUAD>(kp, grid, s, dev);
  if (alibi) return launch_variant<D, true, false, PAIR, QUAD>(kp, grid, s, dev);
  if (softcap) return launch_variant<D, false, true, PAIR, QUAD>(kp, grid, s, dev);
  return launch_variant<D, false, false, PAIR, QUAD>(kp, grid, s, dev);
}

}  // namespace

namespace {
// The same expression as the forward kernel's default slope, in the same
// translation unit and with the same compiler flags.
__global__ void default_alibi_slopes_kernel(float* dst, int H) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h < H) dst[h] = exp2f(-8.0f * (float)(h + 1) / (float)H);
}
}  // namespace

cudaError_t launch_default_alibi_slopes(float* dst, int H, cudaStream_t stream) {
  default_alibi_slopes_kernel<<<(H + 127) / 128, 128, 0, stream>>>(dst, H);
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd(const FwdArgs& a, cudaStream_t stream) {
  KParams kp;
  memset(&kp, 0, sizeof(kp));
  const bool pair = a.cta_pair != 0 && a.D == 128;
  if (pair && a.tpe != kTilesPerQuad) return cudaErrorInvalidValue;
  if (!make_map(&kp.tmap_q, a.q, a.D, a.S_q, a.B * a.H) ||
      !make_map(&kp.tmap_k, a.k, a.D, a.S_k, a.B * a.H_kv) ||
      !make_map(&kp.tmap_v, a.v, a.D, a.S_k, a.B * a.H_kv) ||
      (pair && !make_map(&kp.tmap_kh, a.k, a.D, a.S_k, a.B * a.H_kv, kTileN / 2)) ||
      (!pair && (a.score_flags & (ATTN_SCORE_SOFTCAP | ATTN_SCORE_ALIBI | ATTN_SCORE_RELBIAS)) &&
       !make_map(&kp.tmap_o, a.out, a.D, a.S_q, a.B * a.H)))
    return cudaErrorInvalidValue;
  BlockMaskGeom g = block_mask_geom(a.B, a.S_q, a.S_k, a.mask.flags, a.tpe);
  kp.out = reinterpret_cast<__nv_bfloat16*>(a.out);
  kp.lse = a.lse;
  kp.B = a.B;
  kp.H = a.H;
  kp.H_kv = a.H_kv;
  kp.S_q = a.S_q;
  kp.S_k = a.S_k;
  kp.group = a.H / a.H_kv;
  kp.scale = a.scale;
  kp.scale_log2 = a.scale * kLog2e;
  kp.mask_flags = a.mask.flags;
  kp.window = a.mask.window;
  kp.q_offset = a.mask.q_offset;
  kp.doc_ids = a.mask.doc_ids;
  kp.prefix_len = a.mask.prefix_len;
  kp.alibi_slopes = a.alibi_slopes;
  kp.alibi_on = (a.score_flags & ATTN_SCORE_ALIBI) ? 1 : 0;
  kp.rel_bias = (a.score_flags & ATTN_SCORE_RELBIAS) ? a.rel_bias : nullptr;
  kp.rel_max = a.rel_max;
  kp.blocks = a.mask.blocks;
  kp.softcap = (a.score_flags & ATTN_SCORE_SOFTCAP) ? a.softcap : 0.f;
  const char* base = reinterpret_cast<const char*>(a.block_mask);
  kp.hdr = reinterpret_cast<const BlockMaskHeader*>(base);
  kp.order = reinterpret_cast<const int32_t*>(base + g.order_off);
  kp.cnt = reinterpret_cast<const int32_t*>(base + g.cnt_off);
  kp.list = reinterpret_cast<const uint32_t*>(base + g.list_off);
  if (g.doc_off != 0) {
    kp.doc_lo = reinterpret_cast<const int32_t*>(base + g.doc_off);
    kp.doc_hi = kp.doc_lo + (size_t)g.bm * a.S_k;
  }
  kp.nK = g.nK;
  kp.nP = g.nP;
  kp.bm = g.bm;
  kp.n_entries = g.n_entries;
  const int sub = pair ? 1 : g.tpe / kTilesPerItem;  // work items per entry
  kp.n_items = g.n_entries * (a.B / g.bm) * a.H * sub;
  kp.status = a.status;
  kp.tau = a.rescale_threshold;
  kp.budget_ns = (uint64_t)(a.wait_budget_ms * 1.0e6);
  kp.debug_stall = a.debug_stall;
  if (kp.softcap > 0.f) {
    // u = kk v: the raw score (kk = scale / cap), or y with position biases
    // (the bias variant's pre-cap value, kk = 1 / (2 log2 e))
    const bool biased = (a.score_flags & (ATTN_SCORE_ALIBI | ATTN_SCORE_RELBIAS)) != 0;
    const double l2e = 1.4426950408889634;
    const double kk = biased ? 1.0 / (2.0 * l2e) : (double)a.scale / (double)kp.softcap;
    const double C = (double)kp.softcap * l2e;
    const double r[3] = {ATTN_TANH_POLY_R0, ATTN_TANH_POLY_R1, ATTN_TANH_POLY_R2};
    double kpow = kk;
    bool normal = true;
    for (int i = 0; i < 3; ++i) {
      kp.tq[i] = (float)(C * r[i] * kpow);
      normal = normal && fabsf(kp.tq[i]) >= FLT_MIN && isfinite(kp.tq[i]);
      kpow *= kk * kk;
    }
    // the polynomial path needs normal coefficients; otherwise every tile
    // takes the exp2 / reciprocal formula
    kp.tlim = normal ? (float)(ATTN_TANH_POLY_U0 / kk) : -1.0f;
    kp.ty = biased ? 1.0f : (float)(2.0 * l2e * kk);
  }
  kp.poly_chunks = (int)lrintf(a.poly_fraction * 8.0f);
  if (kp.poly_chunks < 0) kp.poly_chunks = 0;
  if (kp.poly_chunks > 8) kp.poly_chunks = 8;

  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  static std::atomic<int> sm_count[kLaunchCacheDevices];
  if (dev >= 0 && dev < kLaunchCacheDevices) sms = sm_count[dev].load(std::memory_order_relaxed);
  if (sms == 0) {
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < kLaunchCacheDevices) sm_count[dev].store(sms, std::memory_order_relaxed);
  }
  int grid = a.num_ctas > 0 ? a.num_ctas : sms;
  const int per_unit = pair ? 2 : 1;  // CTAs per work unit
  if (grid > kp.n_items * per_unit) grid = kp.n_items * per_unit;
  if (grid < per_unit) grid = per_unit;

  // ALiBi and the bias table share one variant (additive position biases)
  const bool alibi = (a.score_flags & (ATTN_SCORE_ALIBI | ATTN_SCORE_RELBIAS)) != 0;
  const bool softcap = (a.score_flags & ATTN_SCORE_SOFTCAP) != 0;
  const bool quad = g.tpe == kTilesPerQuad;
  if (a.D == 128 && pair)
    return launch_d<128, true, true>(kp, alibi, softcap, grid, stream, dev);
  if (a.D == 128 && !quad)
    return launch_d<128, false, false>(kp, alibi, softcap, grid, stream, dev);
  if (a.D == 64 && quad) return launch_d<64, false, true>(kp, alibi, softcap, grid, stream, dev);
  if (a.D == 64) return launch_d<64, false, false>(kp, alibi, softcap, grid, stream, dev);
  return cudaErrorInvalidValue;  // four-tile masks at D = 128 run on CTA pairs
}

}  // namespace attn
