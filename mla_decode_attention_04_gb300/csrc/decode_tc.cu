// decode_tc.cu -- tensor-core (tcgen05 / TMEM) absorbed-MLA decode, dense and sparse.
//
// Math per (token, head) row, as in "vllm.v1.attention.backends.mla.
// flashattn_mla" (_forward_decode: scores q_nope.kv_c + q_pe.k_pe, values
// kv_c, softmax scale, LSE) with the per-row DCP key limit of the "[Attention]
// add DCP support for FLASH_ATTN_MLA backend" mask tables, or with the
// per-token key lists of sparse MLA.
//
// One CTA per SM walks work units (request or token, row group, KV chunk).
// A unit's NR rows (NR = 16, 32 or 64 (token, head) pairs) share every key,
// so per 64-key tile:
//   S  [128 lanes x 64]  = Q (rows repeated to 128 lanes) . KV^T       (K = 576)
//   O^T[512 x NR]       += KV_c^T (smem, MN-major) . P^T (smem)        (K = 64)
// The first product keeps the 64 keys on the MMA's N side, the second puts
// the 512 latent dims on M and the few rows on N, so neither wastes the
// tensor core on padding for the value product and O^T only needs 4*NR TMEM
// columns next to Q and S (64).  Q sits in TMEM (288 columns) for NR <= 32;
// for NR = 64 its first 192 dims are a shared-memory operand, loaded by TMA
// like a key tile, so that O^T (256 columns) fits.  Bigger units read each
// key tile for more rows: a 64-row unit covers a token of 64 heads, or a
// quarter of a 2-token, 128-head request.  For fp32 outputs P enters the value
// product as two bf16 terms (hi + lo, both accumulated into O^T), so the
// probabilities keep fp32-level precision; for bf16 outputs one bf16 term.
// QK^T and PV are issued by two threads in different warps (one thread
// cannot issue these small MMAs fast enough to keep the tensor pipe busy),
// and S is double-buffered for NR = 16, so the score product of tile j+1
// overlaps the softmax and the value product of tile j.
//
// Warp roles: producer (TMA tile loads through the block table; for sparse,
// 4 warps gathering whole rows with cp.async from the addresses the key-list
// kernel resolved), the QK^T warp (also owns TMEM), four softmax warps (one
// per TMEM lane quarter) that also rescale O^T, zero the value rows of keys
// past the chunk end and write the outputs (a chunk of a split row group as a
// normalised partial with its LSE, merged by the split-merge kernel that runs
// after this one), and the PV warp.  A 3-stage shared-memory ring of 64-key
// tiles (72 KB each; 2 stages for NR = 64) keeps up to 216 KB of KV loads in
// flight per SM; each unit's Q rows take one ring slot ahead of its tiles.  Both variants cut the
// work into balanced contiguous ranges of key tiles, one per CTA (the split
// plan below).  The online softmax rescales O^T lazily: the running reference
// max only moves when a tile's max exceeds it by more than 2^8.
#include <string.h>

#include <type_traits>

#include "common.cuh"
#include "decode_args.h"
#include "decode_kernels.h"
#include "pdl_launch.h"
#include "tc_ptx.cuh"
#include "tma_host.h"

namespace mla {

namespace {

using namespace tc;

constexpr int kChunk = 64 * 128;        // one 64-key x 64-dim bf16 tile, SW128
constexpr int kStageBytes = 9 * kChunk;  // 576 dims
constexpr int kColQ = 0;                 // TMEM columns: Q first
// Where a unit's operands live, by rows per unit NR.
//  * NR = 16, 32: Q in TMEM (9 chunks of 64 dims = 288 columns), S after it;
//    S double-buffered when TMEM has room (NR = 16: 288 + 2*64 + 4*16 = 480
//    columns), so QK^T of tile j+1 runs while the softmax reads S of tile j.
//  * NR = 64: O^T takes 4*64 = 256 columns, so Q's first 3 chunks (dims
//    0-191) are a shared-memory operand (each row twice: TMEM lanes l and
//    l + 64 hold the same row) and only chunks 3-8 sit in TMEM (192
//    columns); S gets the remaining 64.  Shared memory then holds 2 ring
//    stages (not 3) next to the 48 KB of Q and a separate P lo buffer.
template <int NR> struct TmemPlan {
  static constexpr int kQSmemChunks = NR == 64 ? 3 : 0;
  static constexpr int kColS = kColQ + (9 - kQSmemChunks) * 32;  // S buffers [kColS, kColS + 64 SBUF)
  static constexpr int kSBufs = NR == 16 ? 2 : 1;
  static constexpr int kColO = kColS + kSBufs * 64;  // O^T [kColO, kColO + 4 NR)
  static_assert(kColO + 4 * NR <= 512, "TMEM budget");
};
template <int NR, bool KV8 = false> struct Pipe {
  static constexpr int kStages = NR == 64 ? 2 : 3;
  // a unit's Q rows travel through one ring slot, row r at r * kQRowBytes:
  // with room to spare, a 16-byte pad puts consecutive rows in different
  // banks for the softmax warps' row reads (64 padded rows would not fit)
  static constexpr int kQRowBytes = NR == 64 ? kRow * 2 : kRow * 2 + 16;
  static_assert(NR * kQRowBytes <= kStageBytes, "Q slot");
  static constexpr int kQSmemBytes = TmemPlan<NR>::kQSmemChunks * 128 * 128;  // [chunk][128 rows][128 B]
  static constexpr int kPBytes = NR * 128;  // P^T (NR rows x 64 keys bf16, SW128 K-major)
  // P lo sits next to P hi in the stage's k_pe chunk when both fit (8 KB),
  // else in a buffer of its own per stage
  static constexpr bool kPLoInChunk = 2 * kPBytes <= kChunk;
  static constexpr int kPLoBytes = kPLoInChunk ? 0 : kStages * kPBytes;
  static constexpr int kOffQSmem = kStages * kStageBytes;
  static constexpr int kOffPLo = kOffQSmem + kQSmemBytes;
  static constexpr int kOffShared = kOffPLo + kPLoBytes;
  static_assert(!KV8 || NR <= 32, "FP8 caches use units of up to 32 rows");
};
// FP8 caches: a tile's raw codes land in the upper half of the very stage
// they are widened into, as 4 boxes of 128 columns (64 rows x 128 B,
// 128-byte swizzle, 8 KB each, 1024-aligned) and one of the last 64 columns
// (64 rows x 64 B, no swizzle).  Widening part m writes chunks 2m, 2m+1 (part
// 3 also chunk 8): parts 0-2 overwrite only raw parts already widened, part 3
// overwrites its own codes, which every thread reads before any writes.
__host__ __device__ constexpr int raw_part_off(int m) { return 36864 + 8192 * m; }
constexpr int kRawTailOff = 36864 + 4 * 8192;
static_assert(kRawTailOff + 4096 == 9 * 8192, "raw codes end at the stage's end");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// Where a pipeline wait gave up (the workspace header's diagnostic word).
// (2 and 15 are unused: earlier FP8 staging waits, kept so the numbers of
// the others stay stable)
enum WaitSite : int32_t {
  kSiteProducerQ = 1, kSiteProducerStage = 3, kSiteSparseQ, kSiteSparsePart, kSiteQkQ, kSiteQkSFree, kSiteQkFull,
  kSitePvReady, kSiteConvert, kSiteSoftmaxQ, kSiteSoftmaxS, kSiteSoftmaxPv, kSiteSoftmaxUnit
};
// Budget of a wait for copies or MMAs already issued when a role gave up
// (they complete by themselves; the bound only keeps the kernel finite).
constexpr uint64_t kDrainNs = 1000000000ull;

// P^T (NR rows x 64 keys, bf16, SW128 K-major) lives in the k_pe chunk of
// the tile's own stage, free once QK^T of the tile is done: P as bf16 hi at
// offset 0, and for fp32 outputs lo = bf16(P - hi) at offset kPBytes (NR <=
// 32) or in the stage's P lo buffer (NR = 64).
constexpr int kPChunk = 8;  // the k_pe chunk of a stage
constexpr int kMaxStages = 3;
// A stage is filled and freed in 4 parts: part m holds chunks 2m and 2m + 1,
// the dims block 128m..128m+127 that value-product block m reads, and part 3
// also the k_pe chunk (P's home after the score product).  Each part has
// its own full and empty barrier, so the producer refills a stage part by
// part as the value product's blocks complete, and the score product of the
// next tile in the stage starts on its first parts while the last ones
// still load.
constexpr int kParts = 4;
__host__ __device__ constexpr int part_first_chunk(int m) { return 2 * m; }
__host__ __device__ constexpr int part_chunks(int m) { return m == kParts - 1 ? 3 : 2; }

struct TcShared {
  uint64_t full[kMaxStages][kParts];
  uint64_t empty[kMaxStages][kParts];
  uint64_t stg_full[kMaxStages][kParts];  // FP8: a stage part's raw codes have landed
  uint64_t drain[2];  // completion of every MMA of the QK^T / PV thread, at exit
  uint64_t s_full[2], s_free[2], p_ready, pv_done, unit_done, q_ready;
  uint32_t tmem_base;
  int32_t any_rescale[2];
  int32_t wait_ok;  // result of the softmax group's last mbarrier wait
  int32_t conv_ok;  // result of the FP8 converters' last wait for a part's codes
  int32_t prod_ok;  // result of the sparse producer group's last wait
  float alpha[64], inv_l[64];
  // per-tile partial row maxima [tile parity][key slice * NR + row] (the
  // 128 TMEM lanes hold 128 / NR key slices of each of the NR rows)
  float red[2][128];
  float lpart[128];  // partial row sums at the epilogue [key slice * NR + row]
  // split plan of this CTA (written once at the start)
  int64_t plan_lo, plan_hi, plan_W, plan_G, plan_ib;
  int32_t plan_b;  // request holding the range's first item, -1: no work
  ReqFacts plan_f;
  int64_t scan_tmp[16];
};

// 2^x with the hardware ex2 instruction (flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool SPARSE, int NR, bool KV8 = false>
struct Roles {
  // sparse: warps gathering key rows (2 for 64-row units, whose softmax
  // needs the registers a 4-warp CTA could not give it)
  static constexpr int kProducerWarps = SPARSE ? (NR == 64 ? 2 : 4) : 1;
  static constexpr int kMmaWarp = kProducerWarps;          // issues QK^T (and owns TMEM)
  static constexpr int kSoftmaxWarp0 = kProducerWarps + 1;  // four consecutive warps
  static constexpr int kPvWarp = kProducerWarps + 5;        // issues PV
  // FP8 caches: warps widening each FP8 tile to bf16 in its stage
  // (and filling the units' Q slots)
  static constexpr int kConvWarps = KV8 ? 4 : 0;
  static constexpr int kConvWarp0 = kProducerWarps + 6;
  static constexpr int kThreads = (kProducerWarps + 6 + kConvWarps) * 32;
};

// Work unit description, identical for every role.
struct Unit {
  int b, row0, nrows, key0, key1, n_kt;
  int t0;     // dense: first tile of the unit in the request's tile sequence
  int q0, q_len, seq_len, local_len;
  int split, nsplit;
  int cta0;   // dense: CTA holding the pair's first chunk (its counter, its slots)
  int token;  // sparse: the token
};

// What the split plan walks: requests (dense; a pair is a (request, row
// group) over the request's key tiles on the call's shards) or tokens
// (sparse; a pair is a (token, head group) over the token's key list).
template <int NR, bool SPARSE>
struct Source {
  static __device__ __forceinline__ int count(const DecodeArgs& a) { return SPARSE ? a.num_tokens : a.num_requests; }
  // the raw inputs of source i (dense: query_start_loc[i], [i + 1] and
  // seq_lens[i]; sparse: the key count of token i)
  static __device__ __forceinline__ void load(const DecodeArgs& a, int i, int& r0, int& r1, int& r2) {
    if constexpr (SPARSE) {
      r0 = a.list_count[i];
      r1 = r2 = 0;
    } else {
      r0 = a.query_start_loc[i];
      r1 = a.query_start_loc[i + 1];
      r2 = a.seq_lens[i];
    }
  }
  static __device__ __forceinline__ ReqFacts facts(const DecodeArgs& a, int i, int r0, int r1, int r2) {
    if constexpr (SPARSE) {
      ReqFacts f;
      f.ok = true;
      f.q0 = i;
      f.q_len = 1;
      f.seq_len = 0;
      f.local_len = r0;  // keys in the token's list
      f.groups = (a.num_heads + NR - 1) / NR;
      f.nt = (r0 + kKeyTile - 1) / kKeyTile;
      return f;
    } else {
      return request_facts_of(r0, r1, r2, a.num_tokens, a.num_heads, a.dcp_world, a.shard0, a.nshard, NR,
                              !a.noncausal);
    }
  }
};

// Items a source contributes to the split plan: its pairs (row groups;
// with gangs of S > 1 CTAs the pairs share the items, so one) times its key
// tiles plus the unit start-up cost; nothing without keys or rows.
__device__ __forceinline__ int64_t source_items(const ReqFacts& f, int64_t pen, int S) {
  if (f.nt <= 0 || f.groups <= 0) return 0;
  return (S > 1 ? 1 : (int64_t)f.groups) * ((int64_t)f.nt + pen);
}

// The sequence of units of one CTA.  Every (source, row group) pair
// contributes unit_penalty work-free items (the cost of starting a unit)
// followed by its 64-key tiles to one flattened list of W items; CTA c takes
// items [c W / G, (c + 1) W / G), cut at pair boundaries.  With gangs of S
// CTAs (dense calls whose requests have several row groups), a source
// contributes its items once, not once per row group: gang j = c / S takes
// items [j W / G, (j + 1) W / G) (G gangs) and its CTA g = c % S runs row
// group g of each source over them; a pair's chunks are then on CTAs S
// apart.  The CTA found the source holding its first item at start-up
// (plan_cta); the next source's raw inputs are loaded one source ahead and
// turned into facts only when the walk reaches it, so no step of the walk
// waits for a load.  Every role walks the same sequence.
template <int NR, bool SPARSE>
struct UnitIter {
  int64_t i, hi, W, G, ib;  // next item, range end, plan, item base of source b
  int b;
  int S, gg;  // gang size (1: no gangs) and this CTA's row group within its gang
  ReqFacts cur;
  int n0, n1, n2;  // raw inputs of source b + 1

  __device__ __forceinline__ void fetch_next(const DecodeArgs& a) { Source<NR, SPARSE>::load(a, b + 1, n0, n1, n2); }

  __device__ void init(const DecodeArgs& a, const TcShared& sh) {
    S = (!SPARSE && a.gang > 1) ? a.gang : 1;
    gg = (int)blockIdx.x % S;
    if (sh.plan_b < 0) {
      i = hi = 0;
      return;
    }
    i = sh.plan_lo;
    hi = sh.plan_hi;
    W = sh.plan_W;
    G = sh.plan_G;
    b = sh.plan_b;
    ib = sh.plan_ib;
    cur = sh.plan_f;
    if (b + 1 < Source<NR, SPARSE>::count(a)) fetch_next(a);
  }

  __device__ bool next(const DecodeArgs& a, Unit& w) {
    const int64_t pen = a.unit_penalty;
    const int nsrc = Source<NR, SPARSE>::count(a);
    while (true) {
      if (i >= hi) return false;
      const int64_t vlen = (int64_t)cur.nt + pen;
      const int64_t rend = ib + source_items(cur, pen, S);  // end of source b's items
      if (i >= rend) {
        // source b is done (or owns no item): the next one
        if (b + 1 >= nsrc) {
          i = hi;
          return false;
        }
        ib = rend;
        ++b;
        cur = Source<NR, SPARSE>::facts(a, b, n0, n1, n2);
        if (b + 1 < nsrc) fetch_next(a);
        continue;
      }
      // row group holding item i (gangs: this CTA's group, items shared)
      const int g = S > 1 ? gg : (int)quot_floor(i - ib, vlen);
      const int64_t item0 = ib + (S > 1 ? 0 : (int64_t)g * vlen) + pen;
      // the range may start among the items that only carry the pair's
      // start-up cost; a range holding none of its key tiles has no unit
      if (i < item0) i = item0;
      if (i >= hi) return false;
      const int64_t end = min(hi, item0 + cur.nt);
      if (g >= cur.groups) {  // gangs: this source has no row group g
        i = end;
        continue;
      }
      w.token = SPARSE ? b : -1;
      w.b = b;
      w.row0 = g * NR;
      w.nrows = min(NR, cur.q_len * a.num_heads - g * NR);
      w.t0 = (int)(i - item0);
      w.key0 = w.t0 * kKeyTile;
      w.key1 = (int)(end - item0) * kKeyTile;
      if (SPARSE && w.key1 > cur.local_len) w.key1 = cur.local_len;  // the list's end
      w.n_kt = (int)(end - i);
      const int own0 = (int)range_owner(item0, W, G);  // CTA (gangs: gang) of the pair's first tile
      w.cta0 = own0 * S + gg;
      w.nsplit = (int)(range_owner(item0 + cur.nt - 1, W, G) - own0 + 1);
      w.split = (int)blockIdx.x / S - own0;  // the unit's items are this CTA's
      w.q0 = cur.q0;
      w.q_len = cur.q_len;
      w.seq_len = cur.seq_len;
      w.local_len = cur.local_len;
      i = end;
      return true;
    }
  }
};

// Split plan of this CTA, by all its threads before the roles start: W =
// the list length (a block-wide sum over the sources), this CTA's range, and
// the source holding the range's first item (published in sh).  Kept
// to one copy of the scan: the kernel's first instructions are fetched cold
// while they run, so start-up code is kept short.
template <int NR, bool SPARSE>
__device__ __forceinline__ void plan_cta(const DecodeArgs& a, TcShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int B = Source<NR, SPARSE>::count(a);
  const int64_t pen = a.unit_penalty;
  // gangs of S CTAs: a source's items counted once; this CTA plans as gang c / S of gridDim / S
  const int S = (!SPARSE && a.gang > 1) ? a.gang : 1;
  const int64_t me = (int64_t)blockIdx.x / S, nplan = (int64_t)gridDim.x / S;
  const bool single = B <= (int)blockDim.x;  // one chunk of requests: pass 0's facts stay in registers
  ReqFacts f1{};
  int64_t ex1 = 0, lo = 0;
  // pass 0: the list length W and this CTA's range; pass 1: the request
  // whose items contain the range's first item lo
  for (int pass = 0; pass < 2; ++pass) {
    int64_t run = 0;
    for (int base = 0; base < B; base += blockDim.x) {
      const int b = base + tid;
      if (pass == 0 || !single) {
        f1 = ReqFacts{};
        if (b < B) {
          int r0, r1, r2;
          Source<NR, SPARSE>::load(a, b, r0, r1, r2);
          f1 = Source<NR, SPARSE>::facts(a, b, r0, r1, r2);
        }
        // exclusive block scan of the requests' item counts
        const int64_t v = source_items(f1, pen, S);
        int64_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        if (lane == 31) sh.scan_tmp[warp] = x;
        __syncthreads();
        int64_t before = 0, all = 0;
        for (int k = 0; k < nwarps; ++k) {
          const int64_t t = sh.scan_tmp[k];
          if (k < warp) before += t;
          all += t;
        }
        __syncthreads();
        ex1 = run + before + x - v;
        run += all;
      }
      if (pass == 1) {
        const int64_t n = source_items(f1, pen, S);
        if (b < B && n > 0 && ex1 <= lo && lo < ex1 + n) {
          sh.plan_b = b;
          sh.plan_ib = ex1;
          sh.plan_f = f1;
        }
      }
    }
    if (pass == 0) {
      const int64_t W = run;
      const int64_t G = nplan < W ? nplan : (W > 0 ? W : 1);
      const bool has = W > 0 && me < G;
      lo = has ? quot_floor(me * W, G) : 0;
      if (tid == 0) {
        sh.plan_b = -1;
        sh.plan_lo = lo;
        sh.plan_hi = has ? quot_floor((me + 1) * W, G) : 0;
        sh.plan_W = W;
        sh.plan_G = G;
      }
      __syncthreads();
      if (!has) break;
    }
  }
  __syncthreads();
}

// The 16 (32 with P as hi + lo) MMAs of one tile's O^T += V_c^T . P^T (P^T
// hi and lo at descriptors p_hi, p_lo), block m (dims 128m..128m+127) after
// block m - 1, each block's completion committed to the stage part that
// holds its dims (empty[m]), so the producer refills the part while the
// later blocks run.  The first tile of a unit overwrites O^T; the P split
// (hi + lo, for fp32 outputs) doubles the MMAs (they share their A operand,
// which makes the second nearly free).  One rolled copy: the issue rate of
// a thread, not the loop, bounds it.
template <int NR, bool kLoTerm>
__device__ __forceinline__ void issue_pv_tile(uint32_t o0, uint64_t v0, uint64_t p_hi, uint64_t p_lo, uint32_t id_pv,
                                              bool first, bool split, uint64_t* empty) {
#pragma unroll 1
  for (int m = 0; m < kParts; ++m) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t va = v0 + (uint64_t)((2 * m * kChunk + kk * 2048) >> 4);
      mma_ss(o0 + m * NR, va, p_hi + (uint64_t)(kk * 2), id_pv, (first && kk == 0) ? 0u : 1u);
      if (kLoTerm && split) mma_ss(o0 + m * NR, va, p_lo + (uint64_t)(kk * 2), id_pv, 1u);
    }
    mma_commit(&empty[m]);
  }
}

// A tile of a request's sequence: shard index k within the call, tile lt of
// that shard's local keys, the request's local length Lr on that shard.
struct TileLoc {
  int32_t k, lt, Lr;
};

// The cache tensor maps of a dense call, one per shard it covers, and (units
// of 64 rows) the queries' maps.
struct KvMaps {
  CUtensorMap m[kMaxShards];   // bf16 caches; FP8 caches: the 128-column maps
  CUtensorMap m8t[kMaxShards];  // FP8 caches: the maps of the last 64 columns
  CUtensorMap q_nope, q_pe;  // [T H rows][512 | 64 dims] bf16, box 64 rows x 64 dims, 128-byte swizzle
};

__device__ __forceinline__ const CUtensorMap* kv8_tail_map_of(const KvMaps& maps, int k) {
  switch (k) {
    case 0: return &maps.m8t[0];
    case 1: return &maps.m8t[1];
    case 2: return &maps.m8t[2];
    case 3: return &maps.m8t[3];
    case 4: return &maps.m8t[4];
    case 5: return &maps.m8t[5];
    case 6: return &maps.m8t[6];
    default: return &maps.m8t[7];
  }
}

// 4 FP8 E4M3 codes (bytes of x, lowest first) -> 2 bf16x2 words (codes 0,1
// and 2,3), exactly: a code's magnitude bits eeeemmm placed at bits 4-10 of a
// bf16 read as the bf16 2^(e-127) * 1.mmm (or its subnormal 0.mmm * 2^-126 for
// e = 0), so one multiply by 2^120 gives the code's value 2^(e-7) * 1.mmm (or
// m * 2^-9); the sign bit moves to bit 15.  Exact: the products have at most
// 4 significant bits and bf16 arithmetic keeps subnormal operands.  (This GPU
// widens E4M3 to f16 in one instruction, but not to bf16; the f16 route would
// need the bf16 queries in f16 and measured no faster here.)
__device__ __forceinline__ void e4m3x4_to_bf16x2(uint32_t x, uint32_t& lo, uint32_t& hi) {
  const __nv_bfloat162 k = __floats2bfloat162_rn(0x1p120f, 0x1p120f);
  const uint32_t w0 = __byte_perm(x, 0u, 0x4140), w1 = __byte_perm(x, 0u, 0x4342);
  const uint32_t b0 = ((w0 & 0x00800080u) << 8) | ((w0 & 0x007F007Fu) << 4);
  const uint32_t b1 = ((w1 & 0x00800080u) << 8) | ((w1 & 0x007F007Fu) << 4);
  const __nv_bfloat162 r0 = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&b0), k);
  const __nv_bfloat162 r1 = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&b1), k);
  lo = *reinterpret_cast<const uint32_t*>(&r0);
  hi = *reinterpret_cast<const uint32_t*>(&r1);
}

// A 64-row unit's Q rows [grow0, grow0 + 64) as 9 TMA tiles of 64 rows x 64
// dims (128-byte swizzle; rows past the last (token, head) read as zero)
// into one ring slot, chunk c at c * kChunk: the layout of a key tile.
template <int NR>
__device__ __forceinline__ void issue_q_tma(const KvMaps& maps, uint8_t* dst, int64_t grow0, uint64_t* bar) {
  const uint64_t pol = policy_evict_first();
  mbar_arrive_expect_tx(bar, (uint32_t)kStageBytes);
#pragma unroll 1
  for (int c = 0; c < 8; ++c) tma_load_3d(dst + c * kChunk, &maps.q_nope, c * 64, (int32_t)grow0, 0, bar, pol);
  tma_load_3d(dst + 8 * kChunk, &maps.q_pe, 0, (int32_t)grow0, 0, bar, pol);
}

// Address of shard k's map in the kernel's parameter space (static indices).
__device__ __forceinline__ const CUtensorMap* kv_map_of(const KvMaps& maps, int k) {
  switch (k) {
    case 0: return &maps.m[0];
    case 1: return &maps.m[1];
    case 2: return &maps.m[2];
    case 3: return &maps.m[3];
    case 4: return &maps.m[4];
    case 5: return &maps.m[5];
    case 6: return &maps.m[6];
    default: return &maps.m[7];
  }
}

template <int NR, bool SPARSE, bool FUSED, bool KV8>
__global__ void __launch_bounds__(Roles<SPARSE, NR, KV8>::kThreads, 1)
    decode_tc_kernel(const __grid_constant__ KvMaps maps, const __grid_constant__ DecodeArgs a) {
  using R = Roles<SPARSE, NR, KV8>;
  using PP = Pipe<NR, KV8>;
  using TP = TmemPlan<NR>;
  constexpr int kStages = PP::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* kv = base;                           // [kStages][9][kChunk]
  uint8_t* q_smem = base + PP::kOffQSmem;       // NR = 64: Q chunks 0-2 as the QK^T A operand [3][128 rows][128 B]
  uint8_t* p_lo_buf = base + PP::kOffPLo;       // NR = 64: P lo per stage
  TcShared& sh = *reinterpret_cast<TcShared*>(base + PP::kOffShared);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // fp32 outputs get P as bf16 hi + lo (fp32-level probabilities); bf16
  // outputs get bf16 P, already finer than the output rounding
  const bool p_split = a.out_f32 != 0;
  // the same flag as a value the compiler cannot see through (PV issue below)
  bool p_split_rt;
  {
    uint32_t f;
    asm volatile("mov.u32 %0, %1;" : "=r"(f) : "r"(p_split ? 1u : 0u));
    p_split_rt = f != 0u;
  }
  constexpr int SB = TmemPlan<NR>::kSBufs;
  // shards this launch covers: the one-shard instance knows it is one at
  // compile time, so its shard walk folds away
  const int nshard = FUSED ? a.nshard : 1;

  if (warp == R::kMmaWarp) {
    tmem_alloc(&sh.tmem_base, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s)
      for (int m = 0; m < kParts; ++m) {
        mbar_init(&sh.full[s][m], SPARSE ? 32 * R::kProducerWarps : 1);
        mbar_init(&sh.empty[s][m], 1);
      }
    if (KV8)
      for (int b = 0; b < kStages; ++b)
        for (int m = 0; m < kParts; ++m) mbar_init(&sh.stg_full[b][m], 1);
    mbar_init(&sh.drain[0], 1);
    mbar_init(&sh.drain[1], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh.s_full[b], 1);
      mbar_init(&sh.s_free[b], 4);  // one arrival per softmax warp
    }
    mbar_init(&sh.p_ready, 1);
    mbar_init(&sh.pv_done, 1);
    mbar_init(&sh.unit_done, 1);
    mbar_init(&sh.q_ready, 1);
    sh.any_rescale[0] = sh.any_rescale[1] = 0;
    fence_mbar_init();
  }
  if (!SPARSE && warp == R::kMmaWarp && lane < nshard) prefetch_tmap(kv_map_of(maps, lane));
  if (KV8 && warp == R::kMmaWarp && lane < nshard) prefetch_tmap(kv8_tail_map_of(maps, lane));
  if (NR == 64 && warp == R::kMmaWarp && lane == 0) {
    prefetch_tmap(&maps.q_nope);
    prefetch_tmap(&maps.q_pe);
  }
  // The dense decode reads only its inputs until its first global write (a
  // unit's epilogue), so it starts at once, plans its range itself and
  // streams, and waits for the kernels before it in the stream only there;
  // the sparse decode reads the lists kernel's output right away.
  grid_dep_launch();
  if constexpr (SPARSE) grid_dep_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  plan_cta<NR, SPARSE>(a, sh);
  // Every role walks the same units; the first one is found here, in code
  // all warps share (a kernel's instructions are fetched cold as they first
  // run, so each role running its own copy of this step would pay for it
  // again before its first tile).
  UnitIter<NR, SPARSE> it;
  it.init(a, sh);
  Unit w0;
  const bool more0 = it.next(a, w0);
  const uint32_t tmem = sh.tmem_base;
  bool ok = true;
  bool bad_page = false;
  int32_t site = 0;  // where this thread's first wait gave up
  const uint64_t budget = a.wait_ns ? a.wait_ns : 2000000000ull;
  // a pipeline wait: false (and the site noted) once it gave up
  auto wait = [&](uint64_t* bar, uint32_t parity, int32_t where) -> bool {
    if (mbar_wait(bar, parity, budget)) return true;
    if (site == 0) site = where;
    return false;
  };
  // The last phase parity of each ring barrier this thread armed (bit
  // 2 * part + 1: armed, bit 2 * part: parity): at exit the thread waits for
  // those phases, so no copy it issued lands after the CTA is gone.  Only the
  // last arming of a part can be outstanding: re-arming waits for the part's
  // release, which follows its consumption.  Every arming of a part is
  // recorded, a plain arrival too: a parity wait on an older round would
  // alias once the barrier has completed two more.
  uint32_t armed[kMaxStages] = {0, 0, 0}, armed_stg[kMaxStages] = {0, 0, 0};
  auto note_armed = [](uint32_t& word, int m, uint32_t parity) {
    word = (word & ~(3u << (2 * m))) | ((2u | (parity & 1u)) << (2 * m));
  };
  auto drain_armed = [&](uint64_t (*bars)[kParts], const uint32_t* words, int n) {
    for (int s = 0; s < n; ++s)
      for (int m = 0; m < kParts; ++m)
        if ((words[s] >> (2 * m)) & 2u) mbar_wait(&bars[s][m], (words[s] >> (2 * m)) & 1u, kDrainNs);
  };

  if (warp < R::kProducerWarps) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    int q_st = -1;  // FP8: the last Q slot armed and its phase (see below)
    uint32_t q_ph = 0;
    if constexpr (!SPARSE) {
      // The whole warp walks the units; lane l holds the page id of block-
      // table column (cache_col + l), refilled 32 columns at a time, so the
      // block-table reads of 32 pages cost one memory latency.  Lane 0 waits
      // for free stages and issues the TMA loads.
      // a key tile read by one CTA is evicted first; gang members read each
      // tile in turn, so then it stays in L2 at normal priority
      const uint64_t pol = a.gang > 1 ? policy_evict_normal() : policy_evict_first();
      const int ps = a.page_size;
      const int nsub = ps >= kKeyTile ? 1 : kKeyTile / ps;  // pages per tile
      Unit w = w0;
      int cache_b = -1, cache_k = -1, cache_col = 0, my_page = -1;
      // FP8: per stage, the parity of its next key-tile use (Q slots do not
      // touch its raw-code barriers), and the last Q slot armed (stage, phase):
      // the converter warps' arrivals complete the stages' full phases of key
      // tiles, so a Q slot's record is kept apart and dropped once this warp
      // refills that stage (the slot was read then)
      uint32_t kv_ph[kMaxStages] = {0, 0, 0};
      // the unit's Q rows: one slot of the ring (NR <= 32: a bulk copy per
      // row half; NR = 64: 9 TMA tiles of 64 rows x 64 dims)
      auto issue_q = [&](const Unit& u, int st, uint32_t ph) -> bool {
        bool good = true;
        // the slot's bytes all complete on part 0's full barrier; parts 1-3
        // only see an arrival, so every part completes one phase per use
        if (lane == 0) {
          for (int m = 0; m < kParts && good; ++m)
            if (!wait(&sh.empty[st][m], ph ^ 1, kSiteProducerQ)) good = false;
          if (good) {
            if (NR == 64)
              issue_q_tma<NR>(maps, kv + st * kStageBytes, (int64_t)u.q0 * a.num_heads + u.row0, &sh.full[st][0]);
            else
              mbar_arrive_expect_tx(&sh.full[st][0], (uint32_t)u.nrows * (kRow * 2));
            // every part's record moves to this round, so none keeps an
            // older round's parity that the barrier has since passed twice
            if (KV8) {
              q_st = st;
              q_ph = ph;
            } else {
              for (int m = 0; m < kParts; ++m) note_armed(armed[st], m, ph);
            }
            for (int m = 1; m < kParts; ++m) mbar_arrive(&sh.full[st][m]);
          }
        }
        good = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
        if (!good) return false;
        if (NR < 64) {
          uint8_t* qdst = kv + st * kStageBytes;
          for (int r = lane; r < u.nrows; r += 32) {
            const int64_t grow = (int64_t)u.q0 * a.num_heads + u.row0 + r;
            bulk_load(qdst + r * PP::kQRowBytes, a.q_nope + grow * a.q_nope_stride, kNope * 2, &sh.full[st][0]);
            bulk_load(qdst + r * PP::kQRowBytes + kNope * 2, a.q_pe + grow * a.q_pe_stride, kRope * 2,
                      &sh.full[st][0]);
          }
        }
        return true;
      };
      // The Q slot of the CTA's first unit (stage 0, free at the start) is
      // filled by the softmax warps, so this warp goes straight to the key
      // tiles and both start out at once.  This warp is the only one that
      // fills the ring after that (Q slots, key tiles, FP8 codes), one
      // position at a time in ring order, each after the release of the
      // round before: a parity wait on a stage's empty barrier can then never
      // see a round two ahead of the one it waits for.
      bool first = true;
      for (bool more = more0; ok && more; more = it.next(a, w)) {
        if (w.n_kt > 0) {
          if (first) {
            first = false;
          } else if (!issue_q(w, stage, phase)) {
            ok = false;
            break;
          }
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        ShardCursor cur_sh;
        cur_sh.start(w.seq_len, a.dcp_world, a.shard0);
        cur_sh.seek(w.t0, w.seq_len, a.dcp_world, a.shard0, nshard);
        // the current shard's block table, page count and tensor map, picked
        // with static indices when the unit's tiles move to another shard
        const int32_t* bt = pick_shard(a.bts, cur_sh.k);
        int64_t nblk = pick_shard(a.nblocks, cur_sh.k);
        const CUtensorMap* map = kv_map_of(maps, cur_sh.k);
        for (int kt = 0; kt < w.n_kt && ok; ++kt) {
          // tile t of the request's sequence: a tile of shard cur_sh.k's local keys
          if (cur_sh.seek(w.t0 + kt, w.seq_len, a.dcp_world, a.shard0, nshard)) {
            bt = pick_shard(a.bts, cur_sh.k);
            nblk = pick_shard(a.nblocks, cur_sh.k);
            map = kv_map_of(maps, cur_sh.k);
          }
          const TileLoc loc{cur_sh.k, w.t0 + kt - cur_sh.t_begin, cur_sh.Lr};
          const int k = loc.lt * kKeyTile;
          int pages[kKeyTile / 8];
          int nvalid = 0;
#pragma unroll 1
          for (int i = 0; i < nsub; ++i) {
            const int j = k + i * ps;  // first key of this page's part of the tile
            const int col = j / ps;
            if (w.b != cache_b || loc.k != cache_k || col < cache_col || col >= cache_col + 32) {
              cache_b = w.b;
              cache_k = loc.k;
              cache_col = col;
              const int c2 = col + lane;
              const int last_col = (loc.Lr - 1) / ps;
              my_page = (c2 <= last_col && c2 < a.bt_stride) ? bt[(int64_t)w.b * a.bt_stride + c2] : -1;
            }
            const int page = __shfl_sync(0xffffffffu, my_page, col - cache_col);
            pages[i] = -1;
            if (j < loc.Lr) {
              if (page < 0 || page >= nblk || col >= a.bt_stride) {
                bad_page = true;  // recorded at the end, once the status word is this call's
              } else {
                pages[i] = page;
                ++nvalid;
              }
            }
          }
          if (KV8) {
            // FP8: the tile's codes into the upper half of its own stage once
            // the stage's previous round is released (all four parts: the
            // converter widens over the whole stage); the converter warps
            // widen part m into the stage's part m
            if (lane == 0) {
              uint8_t* dst = kv + stage * kStageBytes;
              const uint32_t rows = ps >= kKeyTile ? kKeyTile : ps;
              const int off = ps >= kKeyTile ? k % ps : 0;
              const CUtensorMap* tmap = kv8_tail_map_of(maps, loc.k);
              for (int m = 0; m < kParts && ok; ++m)
                if (!wait(&sh.empty[stage][m], phase ^ 1, kSiteProducerStage)) ok = false;
              if (ok && stage == q_st) q_st = -1;  // that Q slot was read: its copies are in
              for (int m = 0; m < kParts && ok; ++m) {
                mbar_arrive_expect_tx(&sh.stg_full[stage][m],
                                      (uint32_t)(nvalid * rows * (m == kParts - 1 ? 128 + 64 : 128)));
                note_armed(armed_stg[stage], m, kv_ph[stage]);
                for (int i = 0; i < nsub; ++i) {
                  if (pages[i] < 0) continue;
                  tma_load_3d(dst + raw_part_off(m) + i * ps * 128, map, m * 128, off, pages[i],
                              &sh.stg_full[stage][m], pol);
                  if (m == kParts - 1)
                    tma_load_3d(dst + kRawTailOff + i * ps * 64, tmap, 512, off, pages[i], &sh.stg_full[stage][m],
                                pol);
                }
              }
            }
            kv_ph[stage] ^= 1;
          } else if (lane == 0) {
            // part by part, each as soon as the value product frees it
            uint8_t* dst = kv + stage * kStageBytes;
            const uint32_t rows = ps >= kKeyTile ? kKeyTile : ps;
            const int off = ps >= kKeyTile ? k % ps : 0;
            for (int m = 0; m < kParts; ++m) {
              if (!wait(&sh.empty[stage][m], phase ^ 1, kSiteProducerStage)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&sh.full[stage][m], (uint32_t)(nvalid * rows * 128 * part_chunks(m)));
              note_armed(armed[stage], m, phase);
              for (int i = 0; i < nsub; ++i)
                if (pages[i] >= 0)
                  for (int c = part_first_chunk(m); c < part_first_chunk(m) + part_chunks(m); ++c)
                    tma_load_3d(dst + c * kChunk + i * ps * 128, map, c * 64, off, pages[i], &sh.full[stage][m],
                                pol);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
    } else {
      // sparse: the producer warps gather 64 rows x 72 16-byte pieces per
      // tile with cp.async; warp pw copies keys [KW pw, KW pw + KW), one row at a time
      // with all its lanes (a row's 72 pieces in 3 instructions of
      // consecutive 16-byte pieces: every instruction reads whole 128-byte
      // lines), so the memory system sees line-sized requests, not one
      // 16-byte request per thread and piece.
      constexpr int KW = kKeyTile / R::kProducerWarps;  // keys per producer warp: 16 or 32
      const int pw = warp;            // producer warp
      const int pt = threadIdx.x;     // producer thread
      // one thread waits, a named barrier hands the verdict to every producer
      // thread, so all of them take the same path (and the count-based full
      // barriers see every arrival or none)
      auto prod_wait = [&](uint64_t* bar, uint32_t parity, int32_t where) -> bool {
        if (pt == 0) sh.prod_ok = wait(bar, parity, where) ? 1 : 0;
        named_bar_sync(3, 32 * R::kProducerWarps);
        const bool r = sh.prod_ok != 0;
        named_bar_sync(3, 32 * R::kProducerWarps);
        if (r) mbar_wait(bar, parity, kDrainNs);  // every thread observes the phase (returns at once)
        return r;
      };
      Unit w = w0;
      for (bool more = more0; ok && more; more = it.next(a, w)) {
        if (w.n_kt > 0) {
          // the unit's Q rows: one slot of the ring, a bulk copy per row half
          // by thread r (64-row units: 9 TMA tiles by thread 0); every
          // producer thread arrives (the stage's full barrier counts them),
          // thread 0 with the byte count
          bool free_ok = true;
          for (int m = 0; m < kParts; ++m)
            if (!prod_wait(&sh.empty[stage][m], phase ^ 1, kSiteSparseQ)) free_ok = false;
          if (!free_ok) { ok = false; break; }
          uint8_t* qdst = kv + stage * kStageBytes;
          const int64_t grow0 = (int64_t)w.token * a.num_heads + w.row0;
          if (NR < 64 && pt < w.nrows) {
            const int64_t grow = grow0 + pt;
            bulk_load(qdst + pt * PP::kQRowBytes, a.q_nope + grow * a.q_nope_stride, kNope * 2, &sh.full[stage][0]);
            bulk_load(qdst + pt * PP::kQRowBytes + kNope * 2, a.q_pe + grow * a.q_pe_stride, kRope * 2,
                      &sh.full[stage][0]);
          }
          if (pt == 0) {
            if (NR == 64) issue_q_tma<NR>(maps, qdst, grow0, &sh.full[stage][0]);
            else mbar_arrive_expect_tx(&sh.full[stage][0], (uint32_t)w.nrows * (kRow * 2));
          } else {
            mbar_arrive(&sh.full[stage][0]);
          }
          // every part's record moves to this round (parts 1-3: a plain
          // arrival), so none keeps an older round's parity
          for (int m = 0; m < kParts; ++m) note_armed(armed[stage], m, phase);
          for (int m = 1; m < kParts; ++m) mbar_arrive(&sh.full[stage][m]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        const int64_t* rows = a.key_rows + (int64_t)w.token * a.list_stride;
        for (int kt = 0; kt < w.n_kt && ok; ++kt) {
          const int k0 = w.key0 + kt * kKeyTile + pw * KW;
          // lane l (< KW) fetches the row address of key k0 + l
          const int64_t my_row = (lane < KW && k0 + lane < w.key1) ? rows[k0 + lane] : 0;
          uint8_t* dst = kv + stage * kStageBytes;
          // part by part, each as soon as the value product frees it: the
          // part's 16 or 24 pieces of each of the warp's rows, consecutive
          // lanes taking consecutive pieces of a row (whole 128-byte lines)
#pragma unroll
          for (int m = 0; m < kParts; ++m) {
            if (!ok || !prod_wait(&sh.empty[stage][m], phase ^ 1, kSiteSparsePart)) {
              ok = false;
              break;
            }
            constexpr int kPieces[kParts] = {16, 16, 16, 24};
            const int np = kPieces[m], p0 = part_first_chunk(m) * 8;
#pragma unroll 4
            for (int idx = lane; idx < KW * np; idx += 32) {
              const int kk = idx / np, piece = p0 + idx % np;
              const int key = pw * KW + kk;
              const int64_t row = __shfl_sync(0xffffffffu, my_row, kk);
              // a key past the list's end copies no byte (its row is zero-filled)
              const char* src = row != 0 ? reinterpret_cast<const char*>(row) : reinterpret_cast<const char*>(a.kv);
              const uint32_t nbytes = row != 0 ? 16u : 0u;
              const int cc = piece >> 3, within = piece & 7;
              const uint32_t d = smem_u32(dst + cc * kChunk + key * 128 + ((within ^ (key & 7)) << 4));
              asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src + piece * 16),
                           "r"(nbytes)
                           : "memory");
            }
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(&sh.full[stage][m]))
                         : "memory");
            note_armed(armed[stage], m, phase);
          }
          if (!ok) break;
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
    // exit: every copy this thread issued has landed (its armed phases done)
    drain_armed(sh.full, armed, kStages);
    if (KV8) {
      drain_armed(sh.stg_full, armed_stg, kStages);
      if (lane == 0 && q_st >= 0) mbar_wait(&sh.full[q_st][0], q_ph, kDrainNs);
    }
  } else if (warp == R::kMmaWarp || warp == R::kPvWarp) {
    // --------------------------------------------------------------- MMA
    // One thread cannot issue tcgen05.mma fast enough to keep the tensor
    // pipe busy with these small shapes, so QK^T and PV have an issuing
    // thread each (in different warps); each commits its own MMAs.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, j = 0, q_ph = 0;
      const uint32_t id_qk = idesc_bf16_f32(128, 64, 0, 0);
      const uint32_t id_pv = idesc_bf16_f32(128, NR, 1, 0);
      Unit w = w0;
      // Descriptors are linear in the start address (its field is addr >> 4
      // and every address here is below 256 KB), so each operand is a base
      // descriptor plus a constant offset in 16-byte units: the issue loops
      // below are fully unrolled with no descriptor arithmetic per MMA.
      const uint32_t kv0 = smem_u32(kv);
      const uint64_t d_kv = smem_desc_sw128(kv0, 16, 1024);                 // K-major KV rows (QK^T B)
      const uint64_t d_v = smem_desc_sw128(kv0, 8192, 1024);                // MN-major kv_c (PV A)
      const uint64_t d_p = smem_desc_sw128(kv0 + kPChunk * kChunk, 16, 1024);  // P^T hi (PV B)
      // P^T lo: next to hi in the k_pe chunk, or in the stage's own buffer
      const uint64_t d_plo = PP::kPLoInChunk ? d_p + (uint64_t)(PP::kPBytes >> 4)
                                             : smem_desc_sw128(smem_u32(p_lo_buf), 16, 1024);
      constexpr uint64_t kPLoStageUnits = PP::kPLoInChunk ? (kStageBytes >> 4) : (PP::kPBytes >> 4);
      const uint64_t d_q = smem_desc_sw128(smem_u32(q_smem), 16, 1024);  // Q chunks 0-2 (QK^T A, NR = 64)
      constexpr uint64_t kStageUnits = kStageBytes >> 4;
      if (warp == R::kMmaWarp) {
        // S(j) = Q . KV(j)^T into S buffer j % SB as soon as tile j has
        // landed and the softmax has copied S(j - SB) out of that buffer.
        for (bool more = more0; ok && more; more = it.next(a, w)) {
          if (w.n_kt == 0) continue;
          if (++stage == kStages) { stage = 0; phase ^= 1; }  // the unit's Q slot
          if (!wait(&sh.q_ready, q_ph, kSiteQkQ)) { ok = false; break; }
          q_ph ^= 1;
          tc_fence_after();
          for (int kt = 0; kt < w.n_kt; ++kt, ++j) {
            const int sb = j % SB;
            if (!wait(&sh.s_free[sb], ((j / SB) & 1) ^ 1, kSiteQkSFree)) {
              ok = false;
              break;
            }
            const uint64_t b0 = d_kv + (uint64_t)stage * kStageUnits;
            const uint32_t s_col = tmem + TP::kColS + sb * 64;
            // the tile's parts in order, each once it has landed
#pragma unroll
            for (int c = 0; c < 9; ++c) {
              if (c < 8 && (c & 1) == 0) {
                if (!wait(&sh.full[stage][c >> 1], phase, kSiteQkFull)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
              }
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bd = b0 + (uint64_t)(c * (kChunk >> 4) + kk * 2);
                const uint32_t acc = (c | kk) != 0;
                if (c < TP::kQSmemChunks)  // A = Q chunk c in shared memory (128 rows of 128 B)
                  mma_ss(s_col, d_q + (uint64_t)(c * (16384 >> 4) + kk * 2), bd, id_qk, acc);
                else  // A = Q chunk c in TMEM
                  mma_ts(s_col, tmem + kColQ + ((c - TP::kQSmemChunks) * 4 + kk) * 8, bd, id_qk, acc);
              }
            }
            if (!ok) break;
            mma_commit(&sh.s_full[sb]);
            if (++stage == kStages) { stage = 0; phase ^= 1; }
          }
        }
      } else {
        // O^T += V_c(j)^T . P(j)^T once the softmax has written P(j); its
        // completion frees the ring stage (QK^T(j), the stage's other
        // reader, completed before the softmax saw S(j)).
        for (bool more = more0; ok && more; more = it.next(a, w)) {
          if (w.n_kt == 0) continue;
          if (++stage == kStages) stage = 0;  // the unit's Q slot
          for (int kt = 0; kt < w.n_kt; ++kt, ++j) {
            if (!wait(&sh.p_ready, j & 1, kSitePvReady)) { ok = false; break; }
            tc_fence_after();
            const uint64_t v0 = d_v + (uint64_t)stage * kStageUnits;
            const uint64_t p0 = d_p + (uint64_t)stage * kStageUnits;
            const uint64_t p1 = d_plo + (uint64_t)stage * kPLoStageUnits;
            const uint32_t o0 = tmem + TP::kColO;
            // bf16 outputs: hi only, issued back to back; fp32 outputs: the
            // lo MMAs behind a per-step test of the call's flag, which paces
            // them against the score MMAs sharing the tensor pipe (measured:
            // with the test folded away, long context ran 8 % slower)
            if (p_split) issue_pv_tile<NR, true>(o0, v0, p0, p1, id_pv, kt == 0, p_split_rt, sh.empty[stage]);
            else issue_pv_tile<NR, false>(o0, v0, p0, p1, id_pv, kt == 0, false, sh.empty[stage]);
            mma_commit(&sh.pv_done);
            if (kt + 1 == w.n_kt) mma_commit(&sh.unit_done);
            if (++stage == kStages) stage = 0;
          }
        }
      }
      // exit: every MMA this thread issued has completed (TMEM is freed and
      // the stages' memory is reused only after that)
      mma_commit(&sh.drain[warp == R::kMmaWarp ? 0 : 1]);
      mbar_wait(&sh.drain[warp == R::kMmaWarp ? 0 : 1], 0, kDrainNs);
    }
  } else if (KV8 && warp >= R::kConvWarp0) {
    // ---------------------------------------------------------- FP8 widen
    // Each part of a tile's codes (in the upper half of the tile's own stage)
    // becomes the same part of the stage in bf16, in the 128-byte-swizzled
    // chunk layout the bf16 path's TMA writes, part by part so that the score
    // product starts on a tile's first chunks while its last ones widen.
    // Thread ct of the 128 takes row ct / 2 and half ct & 1 of the part's 128
    // code columns (4 pieces of 16 codes -> 8 bf16 pieces), and of the last
    // part's 64 tail columns (2 pieces -> 4 bf16 pieces).  Parts 0-2 write
    // over codes already widened only; part 3 writes over its own codes, so
    // every thread loads all of part 3 before a barrier and writes after it.
    // One thread waits for a part's codes, a named barrier hands the verdict
    // to the others, each of which then observes the completed phase.  The
    // producer waited for the stage's release before loading the codes, so
    // these warps wait for nothing else (they only widen in place; they fill
    // no ring slot).
    const int ct = (int)threadIdx.x - R::kConvWarp0 * 32;
    const int r = ct >> 1, h = ct & 1;
    int stage = 0;
    uint32_t kv_ph[kMaxStages] = {0, 0, 0};  // per stage: parity of its next key-tile use
    Unit w = w0;
    auto widen = [&](const uint4& x, uint8_t* drow, int p0, int p1) {
      uint32_t o[8];
      e4m3x4_to_bf16x2(x.x, o[0], o[1]);
      e4m3x4_to_bf16x2(x.y, o[2], o[3]);
      e4m3x4_to_bf16x2(x.z, o[4], o[5]);
      e4m3x4_to_bf16x2(x.w, o[6], o[7]);
      *reinterpret_cast<uint4*>(drow + ((p0 ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<uint4*>(drow + ((p1 ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
    };
    for (bool more = more0; ok && more; more = it.next(a, w)) {
      if (w.n_kt == 0) continue;
      if (++stage == kStages) stage = 0;  // the unit's Q slot
      for (int kt = 0; kt < w.n_kt && ok; ++kt) {
        uint8_t* st_base = kv + stage * kStageBytes;
        for (int m = 0; m < kParts; ++m) {
          if (ct == 0) sh.conv_ok = wait(&sh.stg_full[stage][m], kv_ph[stage], kSiteConvert) ? 1 : 0;
          named_bar_sync(2, 128);
          if (!sh.conv_ok) {
            ok = false;
            break;
          }
          mbar_wait(&sh.stg_full[stage][m], kv_ph[stage]);  // returns at once
          // columns [128 m, 128 m + 128): code piece v (codes 16v..16v+15)
          // -> bf16 chunk 2m + v / 4, pieces 2 (v % 4) and 2 (v % 4) + 1
          const uint8_t* src = st_base + raw_part_off(m);
          uint4 x[4];
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            x[v4] = *reinterpret_cast<const uint4*>(src + r * 128 + (((4 * h + v4) ^ (r & 7)) << 4));
          uint4 y[2];
          if (m == kParts - 1) {
            // columns [512, 576): tail piece v -> bf16 chunk 8, pieces 2v, 2v + 1
#pragma unroll
            for (int v2 = 0; v2 < 2; ++v2)
              y[v2] = *reinterpret_cast<const uint4*>(st_base + kRawTailOff + r * 64 + (2 * h + v2) * 16);
            named_bar_sync(2, 128);  // every thread has its codes: the writes may cover them
          }
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            widen(x[v4], st_base + (2 * m + h) * kChunk + r * 128, 2 * v4, 2 * v4 + 1);
          if (m == kParts - 1) {
#pragma unroll
            for (int v2 = 0; v2 < 2; ++v2) {
              const int v = 2 * h + v2;
              widen(y[v2], st_base + 8 * kChunk + r * 128, 2 * v, 2 * v + 1);
            }
          }
          fence_proxy_async_smem();
          named_bar_sync(2, 128);
          if (ct == 0) mbar_arrive(&sh.full[stage][m]);
        }
        kv_ph[stage] ^= 1;
        if (++stage == kStages) stage = 0;
      }
    }
  } else {
    // ----------------------------------------------------------- softmax
    const int sw = warp - R::kSoftmaxWarp0;   // 0..3
    const int quarter = warp & 3;             // TMEM lane quarter this warp may access
    const int st_tid = sw * 32 + lane;        // 0..127 within the softmax group
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    // Every unit row is replicated over TPR TMEM lanes (the M = 128 rows of
    // QK^T cost the same whether padded or not), so each softmax thread owns
    // KPT of the 64 keys of one row.  TMEM lane L = 32 q + l (quarter q) holds
    // row L % NR and key slice L / NR: the slice is uniform over a warp (or
    // over each half-warp for NR = 16), so each thread reads just its own
    // columns of S.  The row max is reduced through shared memory; each thread
    // keeps a partial row sum until the unit's epilogue.
    constexpr int TPR = 128 / NR;                 // lanes per row: 8, 4 or 2
    constexpr int KPT = kKeyTile / TPR;           // keys per thread: 8, 16 or 32
    constexpr int RPW = NR >= 32 ? 1 : 32 / NR;   // key slices inside one warp: 2 or 1
    constexpr int CW = NR < 32 ? NR : 32;         // O^T columns per TMEM load (registers)
    const int tl = quarter * 32 + lane;           // this thread's TMEM lane
    const int row = tl % NR;                      // unit row of this lane
    const int kslice = tl / NR;                   // keys [kslice * KPT, + KPT) of the tile
    const int kslice0 = quarter * 32 / NR;        // the warp's first key slice
    const bool row_lead = kslice == 0;            // writes the row's shared values
    // scores in log2 units; an FP8 cache's dequantisation scale multiplies
    // every score (and, in the epilogue, every output)
    const float scale_log2 = a.scale * a.kv_scale * kLog2e;
    const int H = a.num_heads;
    uint32_t j = 0, u_ph = 0;
    int stage = 0;          // ring slot of the next tile (dense: or of the next unit's Q)
    uint32_t sphase = 0;    // its full-barrier parity
    // One thread waits; the named barrier hands its verdict to the group, so
    // the 128 threads always take the same branch (no thread is left at a
    // barrier the others skipped).  Consecutive calls are separated by at
    // least one more group barrier, so the flag is not overwritten early.
    auto group_wait = [&](uint64_t* bar, uint32_t parity, int32_t where) -> bool {
      if (st_tid == 0) sh.wait_ok = wait(bar, parity, where) ? 1 : 0;
      named_bar_sync(1, 128);
      const bool r = sh.wait_ok != 0;
      tc_fence_after();
      return r;
    };
    // global (token, head) row index of row n of unit u
    auto grow_of = [&](const Unit& u, int n) -> int64_t {
      if constexpr (SPARSE) return (int64_t)u.token * H + u.row0 + n;
      else return (int64_t)u.q0 * H + u.row0 + n;
    };
    // the first unit's Q slot (stage 0, first round), filled from here when
    // dense: drained at exit if no load_q consumed it
    bool q0_armed = false, q0_consumed = false;
    // Q rows of unit u into TMEM, then q_ready.  Called once every QK^T
    // issued so far is complete (the softmax has read all their S).
    auto load_q = [&](const Unit& u) -> bool {
      // Q row of this lane -> its TMEM lane: 32 columns (64 bf16) per chunk
      // (the TPR lanes of a row read the same addresses); NR = 64: chunks 0-2
      // into the shared-memory A operand instead, at row tl
      const bool have = row < u.nrows;
      // the rows are in this unit's Q slot of the ring
      if (!group_wait(&sh.full[stage][0], sphase, kSiteSoftmaxQ)) return false;
      if (stage == 0 && sphase == 0) q0_consumed = true;
      mbar_wait(&sh.full[stage][0], sphase);  // every reader observes the phase (returns at once)
      const uint8_t* slot = kv + stage * kStageBytes;
#pragma unroll 1
      for (int c = 0; c < 9; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          // NR <= 32: padded rows; NR = 64: TMA tiles (64 rows x 128 B per
          // chunk, 16-byte pieces swizzled by row & 7)
          const uint8_t* src = NR == 64 ? slot + c * kChunk + row * 128 + ((v ^ (row & 7)) << 4)
                                        : slot + row * PP::kQRowBytes + c * 128 + v * 16;
          const uint4 x = have ? *reinterpret_cast<const uint4*>(src) : make_uint4(0, 0, 0, 0);
          if (c < TP::kQSmemChunks) {
            *reinterpret_cast<uint4*>(q_smem + c * 16384 + tl * 128 + ((v ^ (tl & 7)) << 4)) = x;
          } else {
            r[4 * v] = x.x; r[4 * v + 1] = x.y; r[4 * v + 2] = x.z; r[4 * v + 3] = x.w;
          }
        }
        if (c >= TP::kQSmemChunks) tmem_st<32>(tmem + lane_base + kColQ + (c - TP::kQSmemChunks) * 32, r);
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(1, 128);
      if (st_tid == 0) {
        for (int m = 0; m < kParts; ++m) mbar_arrive(&sh.empty[stage][m]);
        mbar_arrive(&sh.q_ready);
      }
      if (++stage == kStages) { stage = 0; sphase ^= 1; }
      return true;
    };
    Unit w, wn = w0;
    // the split pair whose first chunk this CTA holds (its last unit), for
    // the split-merge kernel: {chunks, first global row, rows, 0}
    int4 desc = make_int4(0, 0, 0, 0);
    bool more = more0;
    if constexpr (!SPARSE) {
      // dense: the first unit's Q slot (stage 0) is filled from here
      if (more && wn.n_kt > 0) {
        q0_armed = true;
        if (NR == 64) {
          if (st_tid == 0) {
            issue_q_tma<NR>(maps, kv, grow_of(wn, 0), &sh.full[0][0]);
            for (int m = 1; m < kParts; ++m) mbar_arrive(&sh.full[0][m]);
          }
        } else {
          if (st_tid == 0) {
            mbar_arrive_expect_tx(&sh.full[0][0], (uint32_t)wn.nrows * (kRow * 2));
            for (int m = 1; m < kParts; ++m) mbar_arrive(&sh.full[0][m]);
          }
          if (st_tid < wn.nrows) {
            const int64_t g = grow_of(wn, st_tid);
            uint8_t* qdst = kv + st_tid * PP::kQRowBytes;
            bulk_load(qdst, a.q_nope + g * a.q_nope_stride, kNope * 2, &sh.full[0][0]);
            bulk_load(qdst + kNope * 2, a.q_pe + g * a.q_pe_stride, kRope * 2, &sh.full[0][0]);
          }
        }
      }
    }
    if (more && wn.n_kt > 0 && !load_q(wn)) ok = false;
    while (ok && more) {
      w = wn;
      more = it.next(a, wn);
      auto grow = [&](int n) -> int64_t { return grow_of(w, n); };
      const bool partial = w.nsplit > 1;
      // sparse: keys [0, kend) of the row's list; dense: the row's global
      // position P and the keys it sees on the current tile's shard (lim),
      // updated when the unit's tiles move to the next shard
      int kend = 0, P_row = -1, lim = 0;
      ShardCursor cur_sh;
      if constexpr (SPARSE) {
        if (row < w.nrows) kend = w.key1;
      } else {
        // the row's global position (non-causal: the request's last key, so
        // the row sees them all)
        if (row < w.nrows) P_row = a.noncausal ? w.seq_len - 1 : w.seq_len - w.q_len + (w.row0 + row) / H;
        cur_sh.start(w.seq_len, a.dcp_world, a.shard0);
        cur_sh.seek(w.t0, w.seq_len, a.dcp_world, a.shard0, nshard);
        lim = P_row >= 0 ? min(visible_keys(P_row, a.dcp_world, a.shard0 + cur_sh.k), cur_sh.Lr) : 0;
      }
      float m_ref = -INFINITY, l_sum = 0.f;

      for (int kt = 0; kt < w.n_kt; ++kt, ++j) {
        // keys of the tile this row sees / that exist (before S is ready:
        // off the score product's path)
        int valid, tile_valid;
        if constexpr (SPARSE) {
          const int kbase = w.key0 + kt * kKeyTile;
          valid = max(0, min(kend - kbase, kKeyTile));
          tile_valid = min(w.key1 - kbase, kKeyTile);
        } else {
          if (cur_sh.seek(w.t0 + kt, w.seq_len, a.dcp_world, a.shard0, nshard))
            lim = P_row >= 0 ? min(visible_keys(P_row, a.dcp_world, a.shard0 + cur_sh.k), cur_sh.Lr) : 0;
          const int kbase = (w.t0 + kt - cur_sh.t_begin) * kKeyTile;
          valid = max(0, min(lim - kbase, kKeyTile));
          tile_valid = min(cur_sh.Lr - kbase, kKeyTile);
        }
        if (!group_wait(&sh.s_full[j % SB], (j / SB) & 1, kSiteSoftmaxS)) { ok = false; break; }
        // this thread's KPT columns of its lane's row of S
        float s[KPT];
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
          uint32_t v[KPT];
          tmem_ld<KPT>(tmem + lane_base + TP::kColS + (j % SB) * 64 + (kslice0 + r) * KPT, v);
          tmem_wait_ld();
          if (kslice - kslice0 == r) {
#pragma unroll
            for (int e = 0; e < KPT; ++e) s[e] = __uint_as_float(v[e]);
          }
        }
        // this warp's part of S is in registers: its lane quarter of the
        // buffer is free for the score product of tile j + SB (each warp
        // arrives once; the row max is exchanged after)
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.s_free[j % SB]);
        // the slice's largest raw score (masked keys -> -inf), as four
        // independent chains; scaled once (the scale is positive)
        if (kslice * KPT + KPT > valid) {  // not every key of the slice visible: a row's last tiles
#pragma unroll
          for (int e = 0; e < KPT; ++e)
            if (kslice * KPT + e >= valid) s[e] = -INFINITY;
        }
        float pm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int e = 0; e < KPT; ++e) pm[e & 3] = fmaxf(pm[e & 3], s[e]);
        const float pmax = fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])) * scale_log2;
        sh.red[j & 1][kslice * NR + row] = pmax;
        tc_fence_before();
        named_bar_sync(1, 128);
        if (st_tid == 0) sh.any_rescale[(j + 1) & 1] = 0;
        {
          float tmax = -INFINITY;
#pragma unroll
          for (int k = 0; k < TPR; ++k) tmax = fmaxf(tmax, sh.red[j & 1][k * NR + row]);
          float alpha = 1.f;
          if (tmax > m_ref + kRescaleThreshold) {  // also the first finite max (m_ref = -inf)
            alpha = fast_exp2(m_ref - tmax);       // 0 when m_ref = -inf
            if (m_ref > -INFINITY && row_lead) sh.any_rescale[j & 1] = 1;
            l_sum *= alpha;
            m_ref = tmax;
          }
          if (row_lead) sh.alpha[row] = alpha;
          // P^T in the k_pe chunk of this tile's stage (QK^T of the tile, its
          // only reader, is complete).  For fp32 outputs P goes in as bf16 hi
          // and lo = bf16(P - hi), so hi + lo carries P to ~2^-16.
          const int roff = (row >> 3) * 1024 + (row & 7) * 128;
          uint8_t* prow = kv + stage * kStageBytes + kPChunk * kChunk + roff;
          uint8_t* prow_lo = PP::kPLoInChunk ? prow + PP::kPBytes : p_lo_buf + stage * PP::kPBytes + roff;
          // P = 2^(s scale_log2 - m_ref) in one fused multiply-add per key
          // (a row with no visible key so far: every s is -inf, P = 0)
          const float neg_m = m_ref > -INFINITY ? -m_ref : -INFINITY;
          float sum4[4] = {0.f, 0.f, 0.f, 0.f};
          // the tile's P, with the hi/lo choice (uniform) outside the loop
          auto write_p = [&](auto split_tag) {
            constexpr bool kSplit = decltype(split_tag)::value;
#pragma unroll
            for (int c8 = 0; c8 < KPT / 8; ++c8) {
              uint32_t hi[4], lo[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float p0 = fast_exp2(fmaf(s[8 * c8 + 2 * e], scale_log2, neg_m));
                const float p1 = fast_exp2(fmaf(s[8 * c8 + 2 * e + 1], scale_log2, neg_m));
                sum4[e] += p0 + p1;
                if constexpr (kSplit) {
                  // hi = P truncated to bf16 (its top 16 bits, one byte permute
                  // for the pair), lo = bf16(P - hi): hi + lo carries P to 2^-16
                  const uint32_t t0 = __float_as_uint(p0) & 0xffff0000u, t1 = __float_as_uint(p1) & 0xffff0000u;
                  hi[e] = __byte_perm(t0, t1, 0x7632);
                  const __nv_bfloat162 l2 =
                      __floats2bfloat162_rn(p0 - __uint_as_float(t0), p1 - __uint_as_float(t1));
                  lo[e] = *reinterpret_cast<const uint32_t*>(&l2);
                } else {
                  const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
                  hi[e] = *reinterpret_cast<const uint32_t*>(&h2);
                }
              }
              const int piece = kslice * (KPT / 8) + c8;  // 16-byte piece (8 keys) of the row
              const int off = (piece ^ (row & 7)) << 4;
              *reinterpret_cast<uint4*>(prow + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
              if constexpr (kSplit) *reinterpret_cast<uint4*>(prow_lo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
          };
          if (p_split) write_p(std::true_type{});
          else write_p(std::false_type{});
          // this thread's part of the row sum (same alpha for every part)
          l_sum += (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
        }
        // value rows of keys past the chunk end: zero them (P is 0 there, and
        // 0 * (garbage) must not reach the accumulator)
        if (tile_valid < kKeyTile) {
          uint8_t* st = kv + stage * kStageBytes;
          const int nz = (kKeyTile - tile_valid) * 64;  // 16-byte pieces over 8 value chunks
          for (int i = st_tid; i < nz; i += 128) {
            const int key = tile_valid + (i >> 6), piece = i & 63;
            *reinterpret_cast<uint4*>(st + (piece >> 3) * kChunk + key * 128 + ((piece & 7) << 4)) =
                make_uint4(0, 0, 0, 0);
          }
        }
        // PV of the previous tile must be complete before O^T is rescaled and
        // before this tile's P is released (waited every tile, in order); the
        // barrier inside group_wait also publishes any_rescale
        if (j > 0) {
          if (!group_wait(&sh.pv_done, (j - 1) & 1, kSiteSoftmaxPv)) { ok = false; break; }
        } else {
          named_bar_sync(1, 128);
        }
        if (sh.any_rescale[j & 1]) {
          // O^T's 4 NR columns, CW per TMEM round trip
#pragma unroll 1
          for (int q = 0; q < 4 * NR / CW; ++q) {
            uint32_t o[CW];
            tmem_ld<CW>(tmem + lane_base + TP::kColO + q * CW, o);
            tmem_wait_ld();
            const int n0 = (q * CW) % NR;
#pragma unroll
            for (int n = 0; n < CW; ++n) o[n] = __float_as_uint(__uint_as_float(o[n]) * sh.alpha[n0 + n]);
            tmem_st<CW>(tmem + lane_base + TP::kColO + q * CW, o);
          }
          tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(1, 128);
        if (st_tid == 0) mbar_arrive(&sh.p_ready);
        if (++stage == kStages) { stage = 0; sphase ^= 1; }
      }
      if (!ok) break;
      // the next unit's Q goes in now, so that its first QK^T overlaps this
      // unit's epilogue
      if (more && wn.n_kt > 0 && !load_q(wn)) {
        ok = false;
        break;
      }

      // ---- epilogue of the unit
      if (w.n_kt > 0) {
        if (!group_wait(&sh.unit_done, u_ph, kSiteSoftmaxUnit)) { ok = false; break; }
        u_ph ^= 1;
      }
      // first global write of this kernel: everything before it in the
      // stream (the previous call's readers of these outputs) has finished
      grid_dep_wait();
      sh.lpart[kslice * NR + row] = l_sum;
      named_bar_sync(1, 128);
      if (row_lead) {
        float lt = 0.f;
#pragma unroll
        for (int k = 0; k < TPR; ++k) lt += sh.lpart[k * NR + row];
        const bool live = lt > 0.f && m_ref > -INFINITY;
        sh.inv_l[row] = live ? a.kv_scale / lt : 0.f;
        if (row < w.nrows) {
          const float lse = live ? (m_ref + __log2f(lt)) * kLn2 : -INFINITY;
          if (partial) a.part_lse[chunk_slot(w.cta0, w.split, NR, it.S) + row] = lse;
          else a.lse[grow(row)] = lse;
        }
      }
      named_bar_sync(1, 128);
      // O^T's 4 NR columns (column m NR + n: dims of block m, row n), 64
      // columns (registers) per TMEM round trip in loads of CW (32 with
      // FP8 caches, whose converter warps leave fewer registers per thread)
      constexpr int PER = (KV8 ? 32 : 64) / CW;
#pragma unroll 1
      for (int q0 = 0; q0 < 4 * NR / CW; q0 += PER) {
        uint32_t o[PER][CW];
        if (w.n_kt > 0) {
#pragma unroll
          for (int p = 0; p < PER; ++p) tmem_ld<CW>(tmem + lane_base + TP::kColO + (q0 + p) * CW, o[p]);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int p = 0; p < PER; ++p)
#pragma unroll
            for (int n = 0; n < CW; ++n) o[p][n] = 0u;
        }
        // rows n0 .. n0 + CW - 1 of one 128-dim block, to one base address
        // at a fixed row stride, 8 values then their 8 stores at a time with
        // no branch between them (a per-value row test and shared-memory
        // load made this a serial chain of ~80 cycles per value)
#pragma unroll
        for (int p = 0; p < PER; ++p) {
          const int col0 = (q0 + p) * CW;
          const int n0 = col0 % NR;
          const int dim = (col0 / NR) * 128 + quarter * 32 + lane;
          const int cnt = min(CW, w.nrows - n0);  // rows of this block the unit has
          const int64_t r0 = partial ? chunk_slot(w.cta0, w.split, NR, it.S) + n0 : grow(n0);
          float* dst32 = (partial ? a.part_o : static_cast<float*>(a.out)) + r0 * kNope + dim;
          __nv_bfloat16* dst16 = static_cast<__nv_bfloat16*>(a.out) + r0 * kNope + dim;
          const bool f32 = partial || a.out_f32;
#pragma unroll
          for (int g = 0; g < CW; g += 8) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(o[p][g + e]) * sh.inv_l[n0 + g + e];
            if (f32) {
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (g + e < cnt) dst32[(int64_t)(g + e) * kNope] = v[e];
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (g + e < cnt) dst16[(int64_t)(g + e) * kNope] = __float2bfloat16_rn(v[e]);
            }
          }
        }
      }
      tc_fence_before();
      if (partial && w.split == 0) desc = make_int4(w.nsplit, (int)grow(0), w.nrows, 0);
      named_bar_sync(1, 128);
    }
    // every CTA publishes its entry (zero chunks: no split pair starts
    // here), after the wait that precedes every global write
    grid_dep_wait();
    if (st_tid == 0) a.split_desc[blockIdx.x] = desc;
    // exit: the first unit's Q copies have landed, consumed or not
    if (q0_armed && !q0_consumed) mbar_wait(&sh.full[0][0], 0, kDrainNs);
  }

  // this kernel completes after the prep kernel, so kernels that wait for it
  // also see the prep kernel's outputs (rows without keys, per-token counts);
  // checks are recorded after it reset the status word
  grid_dep_wait();
  if (!ok) record_wait_timeout(a.hdr, site ? site : 99);
  if (bad_page) record_check(a.hdr, kCheckPageOutOfRange);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == R::kMmaWarp) tmem_dealloc(tmem, 512);
}

template <int NR, bool SPARSE, bool FUSED, bool KV8 = false>
cudaError_t launch_tc(const DecodeArgs& a, const KvMaps& maps, int grid, cudaStream_t stream) {
  const size_t smem = 1024 + Pipe<NR, KV8>::kOffShared + sizeof(TcShared);
  static_assert(1024 + Pipe<NR, KV8>::kOffShared + sizeof(TcShared) <= 232448, "shared memory per CTA");
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<NR, SPARSE, FUSED, KV8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_tc_kernel<NR, SPARSE, FUSED, KV8>, dim3(grid), dim3(Roles<SPARSE, NR, KV8>::kThreads), smem,
                    stream, maps, a);
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeArgs& a, int rows_per_group, bool sparse, int max_units, int num_sms,
                             cudaStream_t stream) {
  if (max_units <= 0) return cudaSuccess;
  if (a.nshard < 1 || a.nshard > kMaxShards || (sparse && a.nshard != 1)) return cudaErrorInvalidValue;
  if (rows_per_group != 16 && rows_per_group != 32 && rows_per_group != 64) return cudaErrorInvalidValue;
  KvMaps maps;
  memset(&maps, 0, sizeof(maps));
  if (a.kv_fp8 && (sparse || rows_per_group > 32)) return cudaErrorInvalidValue;
  for (int k = 0; k < a.nshard; ++k) {
    const bool made = a.kv_fp8 ? make_kv8_tensor_maps(&maps.m[k], &maps.m8t[k], a.kvs[k], a.nblocks[k], a.page_size)
                               : make_kv_tensor_map(&maps.m[k], a.kvs[k], a.nblocks[k], a.page_size);
    if (!made) return cudaErrorInvalidValue;
  }
  if (rows_per_group == 64) {
    const int64_t rows = (int64_t)a.num_tokens * a.num_heads;
    if (!make_query_tensor_map(&maps.q_nope, a.q_nope, rows, kNope, a.q_nope_stride) ||
        !make_query_tensor_map(&maps.q_pe, a.q_pe, rows, kRope, a.q_pe_stride))
      return cudaErrorInvalidValue;
  }
  const int grid = max_units < num_sms ? max_units : num_sms;
  if (sparse) {
    if (rows_per_group == 16) return launch_tc<16, true, false>(a, maps, grid, stream);
    if (rows_per_group == 32) return launch_tc<32, true, false>(a, maps, grid, stream);
    return launch_tc<64, true, false>(a, maps, grid, stream);
  }
  if (a.kv_fp8) {
    if (a.nshard > 1)
      return rows_per_group == 16 ? launch_tc<16, false, true, true>(a, maps, grid, stream)
                                  : launch_tc<32, false, true, true>(a, maps, grid, stream);
    return rows_per_group == 16 ? launch_tc<16, false, false, true>(a, maps, grid, stream)
                                : launch_tc<32, false, false, true>(a, maps, grid, stream);
  }
  if (a.nshard > 1) {
    if (rows_per_group == 16) return launch_tc<16, false, true>(a, maps, grid, stream);
    if (rows_per_group == 32) return launch_tc<32, false, true>(a, maps, grid, stream);
    return launch_tc<64, false, true>(a, maps, grid, stream);
  }
  if (rows_per_group == 16) return launch_tc<16, false, false>(a, maps, grid, stream);
  if (rows_per_group == 32) return launch_tc<32, false, false>(a, maps, grid, stream);
  return launch_tc<64, false, false>(a, maps, grid, stream);
}

}  // namespace mla
