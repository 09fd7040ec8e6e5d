// attn_internal.h -- layouts and parameters shared by the host launcher, the
// block-mask builder and the forward kernel (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attn.h"

namespace attn {

// Tile shape: 128 query rows x 128 keys.  A block-mask entry groups
// kTilesPerItem query tiles (256 rows, the work of one CTA whose two softmax
// warpgroups ping-pong) or, for the CTA-pair forward, kTilesPerQuad query
// tiles (512 rows, the work of one CTA pair).
constexpr int kTileM = 128;
constexpr int kTileN = 128;
constexpr int kTilesPerItem = 2;
constexpr int kTilesPerQuad = 4;

// Tile classes.
enum TileClass : uint32_t { kEmpty = 0, kPartial = 1, kFull = 2 };

// Entry of an entry's key-tile list: key tile index in bits 0..23, then two
// bits of class per query tile of the entry: tile t in bits 24 + 2t .. 25 + 2t.
constexpr uint32_t kListIdxMask = 0x00FFFFFFu;
__host__ __device__ inline uint32_t list_entry(uint32_t kt, uint32_t c0, uint32_t c1) {
  return kt | (c0 << 24) | (c1 << 26);
}
__host__ __device__ inline uint32_t entry_tile(uint32_t e) { return e & kListIdxMask; }
__host__ __device__ inline uint32_t entry_cls(uint32_t e, int t) { return (e >> (24 + 2 * t)) & 3u; }

constexpr uint32_t kBlockMaskMagic = 0x4B4D4241u;  // "ABMK"
constexpr uint32_t kBlockMaskVersion = 2u;

// Device block-mask buffer: header, then order[], cnt[], list[][nK].
struct BlockMaskHeader {
  uint32_t magic;
  uint32_t version;
  int32_t B, S_q, S_k;
  int32_t nQ, nK, nP;       // query tiles, key tiles, entries per mask batch
  int32_t bm;               // batches the mask depends on (B or 1)
  int32_t n_entries;        // bm * nP
  uint32_t mask_flags;
  int32_t window;
  int32_t q_offset;
  int32_t force_partial;
  int32_t uniform;          // 1 when every entry has the same tile count
  int32_t max_cnt;
  uint64_t doc_ptr;         // mask arrays the mask was built from
  uint64_t prefix_ptr;
  uint64_t order_off, cnt_off, list_off;  // byte offsets from the header
  uint64_t total_bytes;
  uint64_t doc_off;         // DOCUMENT: int32 doc_lo[bm][S_k], doc_hi[bm][S_k]
  int32_t docs_sorted;      // 1: every batch's doc ids are non-decreasing
  int32_t tiles_per_entry;  // query tiles per entry: kTilesPerItem or kTilesPerQuad
  uint64_t blocks_ptr;      // BLOCKS: the block map the mask was built from
  uint64_t pad2_;
};
static_assert(sizeof(BlockMaskHeader) % 16 == 0, "header alignment");

struct BlockMaskGeom {
  int tpe;  // query tiles per entry
  int nQ, nK, nP, bm, n_entries;
  size_t order_off, cnt_off, list_off;
  size_t doc_off;   // DOCUMENT only: per-token document key interval
  size_t tile_off;  // DOCUMENT only: smallest / largest id of every 128-token tile
  size_t flag_off;  // DOCUMENT only: int32 "ids out of order" flag per prep block
  int n_flags;
  size_t total;
};

// Tokens per block of the document preparation pass (a multiple of kTileN).
constexpr int kDocPrepTokens = 1024;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Internal mask-flag bit (never accepted from callers): the user block map
// has one map per batch entry, so the block mask depends on the batch.
constexpr uint32_t kMaskBlocksBatched = 1u << 31;
inline bool mask_per_batch(uint32_t mask_flags) {
  return (mask_flags & (ATTN_MASK_DOCUMENT | ATTN_MASK_PREFIX_LM | kMaskBlocksBatched)) != 0;
}

inline BlockMaskGeom block_mask_geom(int B, int S_q, int S_k, uint32_t mask_flags,
                                     int tpe = kTilesPerItem) {
  BlockMaskGeom g;
  g.tpe = tpe;
  g.nQ = (S_q + kTileM - 1) / kTileM;
  g.nK = (S_k + kTileN - 1) / kTileN;
  g.nP = (g.nQ + tpe - 1) / tpe;
  g.bm = mask_per_batch(mask_flags) ? B : 1;
  g.n_entries = g.bm * g.nP;
  g.order_off = align_up(sizeof(BlockMaskHeader), 16);
  g.cnt_off = align_up(g.order_off + sizeof(int32_t) * (size_t)g.n_entries, 16);
  g.list_off = align_up(g.cnt_off + sizeof(int32_t) * (size_t)g.n_entries, 16);
  g.total = align_up(g.list_off + sizeof(uint32_t) * (size_t)g.n_entries * (size_t)g.nK, 16);
  g.doc_off = g.tile_off = g.flag_off = 0;
  g.n_flags = 0;
  if (mask_flags & ATTN_MASK_DOCUMENT) {
    // int32 [bm][S_k] first and last key of each token's document (valid
    // when the ids are non-decreasing), then int32 [bm][nK] id range of each
    // key tile (lo, then hi), then one out-of-order flag per prep block
    g.doc_off = g.total;
    g.tile_off = align_up(g.doc_off + 2 * sizeof(int32_t) * (size_t)g.bm * (size_t)S_k, 16);
    g.flag_off = align_up(g.tile_off + 2 * sizeof(int32_t) * (size_t)g.bm * (size_t)g.nK, 16);
    g.n_flags = g.bm * ((S_k + kDocPrepTokens - 1) / kDocPrepTokens);
    g.total = align_up(g.flag_off + sizeof(int32_t) * (size_t)g.n_flags, 16);
  }
  return g;
}

// Transposed block mask for the key-side backward: for every (mask batch,
// key tile) the non-empty query tiles in ascending order, each entry the
// query tile index in bits 0..23 and its class in bits 24..25.
// Layout: int32 cnt[bm * nK], then uint32 list[bm * nK][nQ].
struct BlockMaskTGeom {
  int nQ, nK, bm, n_entries;
  size_t list_off, total;
};
inline BlockMaskTGeom block_mask_t_geom(int B, int S_q, int S_k, uint32_t mask_flags) {
  BlockMaskTGeom g;
  g.nQ = (S_q + kTileM - 1) / kTileM;
  g.nK = (S_k + kTileN - 1) / kTileN;
  g.bm = mask_per_batch(mask_flags) ? B : 1;
  g.n_entries = g.bm * g.nK;
  g.list_off = align_up(sizeof(int32_t) * (size_t)g.n_entries, 16);
  g.total = align_up(g.list_off + sizeof(uint32_t) * (size_t)g.n_entries * (size_t)g.nQ, 16);
  return g;
}

// Mask parameters as the kernels see them.
struct MaskParams {
  uint32_t flags;
  int32_t window;
  int32_t q_offset;
  int32_t S_q, S_k;
  const int32_t* doc_ids;     // [B][S_k]
  const int32_t* prefix_len;  // [B]
  const uint8_t* blocks;      // [B or 1][nQ][nK] (flags & ATTN_MASK_BLOCKS)
};

// Status codes the device writes (first error wins).
struct DeviceStatus {
  int32_t code;        // attn_status
  int32_t where;       // site id of the failure
  int32_t block;       // blockIdx.x
  int32_t detail;
};

// Launchers (defined in the .cu files, called by the host API).
// tpe: query tiles per entry (kTilesPerItem, or kTilesPerQuad for the
// CTA-pair forward).
cudaError_t launch_build_block_mask(int B, int S_q, int S_k, const MaskParams& mp,
                                    int force_partial, void* dst, cudaStream_t stream,
                                    int tpe = kTilesPerItem);

// Builds the transposed block mask into dst_t from the block mask fwd_mask
// already built (on the same stream) for the same problem.
cudaError_t launch_build_block_mask_t(int B, int S_q, int S_k, const MaskParams& mp,
                                      int force_partial, const void* fwd_mask, void* dst_t,
                                      cudaStream_t stream);

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* lse;
  int B, H, H_kv, S_q, S_k, D;
  float scale;
  MaskParams mask;
  uint32_t score_flags;
  float softcap;
  const float* alibi_slopes;
  const float* rel_bias;       // [H][2 rel_max + 1] (score_flags & ATTN_SCORE_RELBIAS)
  int rel_max;
  const void* block_mask;      // device, built for this call
  int n_entries;
  int bm;
  int nP;
  DeviceStatus* status;        // device
  float rescale_threshold;
  double wait_budget_ms;
  int num_ctas;                // 0 = SM count
  int cta_pair;                // D = 128: CTA-pair kernel (block mask of quads)
  int tpe;                     // query tiles per block-mask entry
  float poly_fraction;
  int debug_stall;             // test hook: MMA issuers wait on a barrier nothing arrives on
};

cudaError_t launch_attn_fwd(const FwdArgs& a, cudaStream_t stream);

// Backward: dQ, dK, dV from Q, K, V, O, LSE and dO (all device pointers).
struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* out;
  const float* lse;
  const void* dout;
  void* dq;
  void* dk;
  void* dv;
  int B, H, H_kv, S_q, S_k, D;
  float scale;
  MaskParams mask;
  uint32_t score_flags;
  float softcap;
  const float* alibi_slopes;
  const float* rel_bias;
  int rel_max;
  const void* block_mask;    // forward block mask, built for this call
  const void* block_mask_t;  // transposed block mask, built for this call
  float* rowstat;            // scratch: [2][B*H][nQ*128] (-LSE in log2 units, -(dO . O))
  DeviceStatus* status;
  double wait_budget_ms;
  int force_partial;
  int debug_stall;  // test hook: 1 stalls the dQ kernel's MMA issuer, 2 the dK/dV kernel's
};

// Bytes of the row-statistics scratch of a backward.
inline size_t bwd_rowstat_bytes(int B, int H, int S_q) {
  const size_t nQ = (size_t)((S_q + kTileM - 1) / kTileM);
  return 2 * sizeof(float) * (size_t)B * (size_t)H * nQ * kTileM;
}

cudaError_t launch_attn_bwd(const BwdArgs& a, cudaStream_t stream);

// dst[h] = the default ALiBi slope of head h of H, bit for bit the value the
// forward kernel computes when it is given no slopes.
cudaError_t launch_default_alibi_slopes(float* dst, int H, cudaStream_t stream);

}  // namespace attn
