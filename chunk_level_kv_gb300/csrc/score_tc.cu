// Tensor-core window scoring (tcgen05 + TMA + TMEM) for bf16 keys, head dim 128.
//
// ChunkKV §4.1 Algorithm 1 steps 1-3 with the probabilities of Kara §2 Eq. (1),
// in the single-pass unit decomposition described in score.cu: each work item
// is one (reuse group, scoring unit, 128-row M tile of the window rows), and one
// persistent launch covers the items of every reuse group.  CTAs claim items in
// order from a counter in the workspace header (the M tiles of a unit go to CTAs
// that start them at about the same time, so their key tiles meet in L2), and a
// CTA that drew short items takes more.  Per item the CTA
//   - has the item's 128 packed window rows (Q) loaded by TMA into shared
//     memory (only when the tile differs from the previous item's),
//   - streams the unit's keys in tiles of 80 through shared memory by TMA,
//   - computes S = Q K^T (128 x 80, fp32) with tcgen05.mma (A and B in shared
//     memory) into one of three TMEM accumulator stages,
//   - lets each of 128 softmax threads own one window row: it reads its row of
//     S from TMEM (16 columns at a time, the next 16 in flight), forms 2^(s*log2(e)/sqrt(d) - R) with R the row maximum of the
//     item's first tile, and sums those per chunk (chunk boundaries are compile
//     time constants for each of the C / gcd(80, C) tile phases), writing one
//     16-bit bin per (chunk, row) and the row's (R, sum) at the end of the item.
// A row whose values would outgrow the first-tile reference by more than 2^23
// switches to the new maximum and rescales what it already wrote.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM owner and MMA
// issuer, warps 2-5 = softmax (warp w reads TMEM lanes 32*(w%4) .. +31).  Two
// CTAs fit on one SM (112 KB shared memory, 256 TMEM columns each).  Every wait
// is bounded: a wait that runs out records an error code in the workspace error
// word, raises a CTA-wide abort flag and the CTA drains and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "fin.cuh"

namespace chunkkv {
namespace tc {

constexpr int kN = 80;                         // keys per tile (MMA N)
constexpr int kD = 128;                        // head dimension
constexpr int kStagesK = 4;                    // key tiles in shared memory (two CTAs of 112 KB per SM)
constexpr int kStagesQ = 1;                    // Q tile in shared memory (reused across items)
// The window-row tile stays in shared memory as MMA operand A (both operands
// there), which leaves all 256 TMEM columns of a CTA to three 80-column fp32
// accumulator stages: the MMAs of two tiles can run ahead of the softmax.
constexpr int kStagesT = 3;                    // accumulator stages in TMEM (80 columns each)
constexpr int kTmemCols = 256;
static_assert(kStagesT >= 2 && kStagesT * kN <= kTmemCols, "TMEM budget");
constexpr int kThreads = 192;                  // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
// Work items handed from the producer to the MMA issuer and the softmax warps
// through a ring in shared memory (the producer claims them from a counter).
constexpr int kItemRing = 2;
constexpr int kPanelQ = 128 * 128;             // one 64-element (128 B) panel of 128 rows
constexpr int kPanelK = kN * 128;              // one 128 B panel of 80 key rows
constexpr int kQBytes = 2 * kPanelQ;           // 32 KB per Q tile
constexpr int kKBytes = 2 * kPanelK;           // 20 KB per K tile
// The dynamic shared window starts 1024-byte aligned (no static shared memory);
// the kernel checks this and reports an error instead of computing on a
// misaligned swizzle pattern.
constexpr int kSmemBytes = kStagesQ * kQBytes + kStagesK * kKBytes + 256;
// barriers, TMEM address, abort flag and item ring in the last 256 bytes
static_assert(8 * (2 * kStagesQ + 2 * kStagesK + 2 * kStagesT + 1 + 2 * kItemRing) + 8 + 4 * kItemRing <= 256,
              "control block");
constexpr uint32_t kIdesc = (1u << 4)                         // D = fp32
                          | (1u << 7) | (1u << 10)           // A = B = bf16
                          | ((uint32_t)(kN >> 3) << 17)      // N
                          | ((uint32_t)(128 >> 4) << 24);    // M
// Rescale threshold of a row sum: just under 2^23 of the reference, (1 - 2^-10)
// 2^(23 - kBinShift) in the scaled values the kernel forms, so that every bin it
// keeps (at most the row sum) rounds to a code inside 16 bits.
constexpr float kBig = (1.0f - 1.0f / 1024.0f) / 9223372036854775808.0f;   // (1 - 2^-10) 2^-63

// One launch scores up to kMaxGroups reuse groups (one layer each): items are
// enumerated group by group, each group with its own key tensor map and its own
// scratch slot (rl, bins at a fixed stride from the first group's).
constexpr int kMaxGroups = 32;

struct TcGeom {
  int32_t B, Hkv, wG, MT, cpu, ku;
  int32_t c;                         // chunk size (the instances with C = 0 read it here)
  int32_t w;                         // window length (for the causal-window limit)
  int32_t G;                         // query heads per KV head
  int32_t q_direct;                  // 1: window rows read from Q_w itself (maps.q[group]), 0: packed (maps.q[0])
  int32_t qm;                        // query heads per 128-row M tile when q_direct (128 / w)
  int32_t qshift;                    // 1: paired sequences (ScoreGeom::pair), sequence b reads window b >> 1
  int32_t items_pg;                  // work items per group: units x M tiles
  int32_t n_items;                   // items_pg x groups of this launch
  int64_t slot_bytes;                // bytes between the scratch slots of consecutive groups
  float alpha;                       // log2(e) / sqrt(d)
  long long timeout;                 // clock64 cycles per wait
};

// Window rows: either one 4-D map per group over that layer's Q_w itself, (d, w,
// Hq, B) with a (64, w, 128 / w, 1) box, whose 128 rows are query heads
// h*G + mt*128/w .. of the M tile with their w window rows each (the packed row
// order; rows past the head's w*G are other heads' or zero-filled and never
// written out), or every group's rows packed by pack_q_kernel in one 2-D map
// (q[0], [rows, 128], row tile `key`) when w does not divide 128.
struct TcMaps {
  CUtensorMap q[kMaxGroups];
  CUtensorMap k[kMaxGroups];         // keys of each group's layer, [T_total, Hkv, 128]
};

// Where work item `item` of a launch lives.
struct Item {
  int grp, unit, mt, b, h, u, nk, ntile, key;
  int64_t tok0;                      // first key row of the unit in the packed varlen key array
};

__device__ __forceinline__ Item decode_item(const TcGeom& g, const SeqTable& st, int item) {
  Item it;
  it.grp = item / g.items_pg;
  const int local = item - it.grp * g.items_pg;
  it.unit = local / g.MT;
  it.mt = local - it.unit * g.MT;
  decode_unit(st, g.Hkv, it.unit, it.b, it.h, it.u);
  const int T = st.cu[it.b + 1] - st.cu[it.b];
  const int k0 = it.u * g.ku;
  it.nk = min(g.ku, T - k0);
  it.ntile = (it.nk + kN - 1) / kN;
  it.key = ((it.grp * g.B + it.b) * g.Hkv + it.h) * g.MT + it.mt;   // packed row tile of its window rows
  it.tok0 = (int64_t)st.cu[it.b] + k0;
  return it;
}

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Test for the completion of the phase with the given parity; a thread whose
// phase is still open is suspended in hardware until the phase completes or
// kSuspendNs nanoseconds pass, instead of spinning on the issue slots that the
// softmax warps of its SM sub-partition need.
constexpr uint32_t kSuspendNs = 1000000;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(bar), "r"(parity), "r"(kSuspendNs) : "memory");
  return ok != 0;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(dst), "l"((uint64_t)map), "r"(bar), "r"(c0), "r"(c1) : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], "
      "[%2];"
      ::"r"(dst), "l"((uint64_t)map), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3) : "memory");
}
// A 3-D tile load with an L2 eviction-priority policy (createpolicy) attached.
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                                 int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%3, %4, %5}], [%2], %6;"
      ::"r"(dst), "l"((uint64_t)map), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy) : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// A bin store that asks L2 to keep the line: the finalisation reads it back soon.
__device__ __forceinline__ void st_keep(bin_t* ptr, float v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.b16 [%0], %1, %2;" ::"l"(ptr), "h"((unsigned short)bin_encode(v)), "l"(policy)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// D (+)= A B^T with A (128 x 16 bf16) in shared memory (matrix descriptor).
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(acc) : "memory");
}
// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                 // leading byte offset (not used by swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset
  d |= (uint64_t)1 << 46;                 // descriptor version
  d |= (uint64_t)2 << 61;                 // 128-byte swizzle
  return d;
}

// 16 consecutive fp32 TMEM columns of this thread's lane (32x32b shape, x16).  The
// registers may only be read after tmem_wait16, which takes them as read-write
// operands so that no use can be scheduled before tcgen05.wait::ld.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])
               :
               : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__host__ __device__ constexpr int gcd_c(int a, int b) { return b == 0 ? a : gcd_c(b, a % b); }

// Shared state of a CTA for bounded waits.
struct Ctl {
  int32_t* err;
  volatile int* abort;
  long long timeout;
};

__device__ __forceinline__ bool wait_bar(const Ctl& ctl, uint32_t bar, uint32_t parity, int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*ctl.abort) return false;
    if (clock64() - t0 > ctl.timeout) {
      atomicCAS(ctl.err, 0, code);
      *ctl.abort = 1;
      return false;
    }
  }
}

// Wait for a phase of an asynchronous operation that this CTA started (a TMA copy
// or a commit of its MMAs) after the CTA gave up: unlike wait_bar it ignores the
// abort flag, since the point is to let that operation land before the shared
// memory and TMEM it writes are released.  Bounded by `limit` cycles; returns
// false if the phase did not complete in time.
__device__ __forceinline__ bool drain_phase(uint32_t bar, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > limit) return false;
  return true;
}

// Cycles a drain waits for one phase (about 50 ms at 2 GHz; a TMA copy or an MMA
// normally lands within microseconds).
constexpr long long kDrainCycles = 100000000LL;

// ---------------------------------------------------------------- softmax side
// Per-row state of the item being processed.
struct RowState {
  float2 negR;     // -(reference exponent), twice (packed operand)
  float2 carry;    // partial sum (two lanes) of a chunk that continues into the next tile
  float l;         // sum of 2^(t - R) over the item's keys so far
};

// Segment SEG (columns 16*SEG .. 16*SEG+15) of a tile whose column 0 has phase PH
// inside its chunk.  Columns are taken in pairs: one packed FMA forms both base-2
// exponents, two MUFU ex2 evaluate them and one packed add accumulates them; the
// pair's two lanes are folded when a chunk ends (compile-time positions).  bin
// points at bins[(gu*cpu + q)*wG + row], q being the unit-local chunk that holds
// the tile's column 0.  C = 1 (token-level chunks) stores every column as a bin.
template <int C, int PH, int SEG, bool MASK, bool STORE>
__device__ __forceinline__ void tile_seg(const uint32_t (&r)[16], float2 alpha2, RowState& s, bin_t* bin, int wG,
                                         int valid, bool write, uint64_t pol) {
  static_assert(C >= 1, "compile-time chunk sizes");
  float2 acc = s.carry;
#pragma unroll
  for (int p = 0; p < 8; ++p) {
    const int c0 = SEG * 16 + 2 * p;
    const float2 x = make_float2(__uint_as_float(r[2 * p]), __uint_as_float(r[2 * p + 1]));
    const float2 t = __ffma2_rn(x, alpha2, s.negR);
    float2 e = make_float2(ex2(t.x), ex2(t.y));
    if (MASK) {
      e.x = (c0 < valid) ? e.x : 0.f;
      e.y = (c0 + 1 < valid) ? e.y : 0.f;
    }
    if constexpr (C == 1) {
      if (STORE && write) {
        st_keep(bin + (size_t)c0 * wG, e.x, pol);
        st_keep(bin + (size_t)(c0 + 1) * wG, e.y, pol);
      }
      s.l += e.x + e.y;
    } else if ((PH + c0 + 1) % C == 0) {        // a chunk ends at the pair's first column
      const float bsum = (acc.x + acc.y) + e.x;
      if (write) st_keep(bin + (size_t)((PH + c0 + 1) / C - 1) * wG, bsum, pol);
      s.l += bsum;
      acc = make_float2(0.f, e.y);
    } else if ((PH + c0 + 2) % C == 0) {        // a chunk ends at the pair's second column
      acc = __fadd2_rn(acc, e);
      const float bsum = acc.x + acc.y;
      if (write) st_keep(bin + (size_t)((PH + c0 + 2) / C - 1) * wG, bsum, pol);
      s.l += bsum;
      acc = make_float2(0.f, 0.f);
    } else {
      acc = __fadd2_rn(acc, e);
    }
  }
  s.carry = acc;
}

// The columns of a tile, software-pipelined: segment SEG is processed while
// segment SEG + 1 is on its way from TMEM (one x16 load in flight beside the
// arithmetic, 32 registers of tile data instead of 80).
template <int C, int PH, int SEG, bool MASK, bool STORE>
__device__ __forceinline__ void tile_segs_pipe(uint32_t taddr, uint32_t (&ra)[16], uint32_t (&rb)[16], float2 alpha,
                                               RowState& s, bin_t* bin, int wG, int valid, bool write, uint64_t pol) {
  if constexpr (SEG < kN / 16) {
    if constexpr (SEG + 1 < kN / 16) tmem_ld16(taddr + 16 * (SEG + 1), rb);
    tile_seg<C, PH, SEG, MASK, STORE>(ra, alpha, s, bin, wG, valid, write, pol);
    if constexpr (SEG + 1 < kN / 16) {
      tmem_wait16(rb);
      tile_segs_pipe<C, PH, SEG + 1, MASK, STORE>(taddr, rb, ra, alpha, s, bin, wG, valid, write, pol);
    }
  }
}

// The same for a chunk size known only at run time (c >= 2): `pos` columns of
// the chunk holding column 0 precede the tile, and the chunk ends are found by
// counting (the count is the same in every lane, so the branches are uniform).
template <bool MASK>
__device__ __forceinline__ void tile_cols_rt(const uint32_t (&r)[kN / 16][16], float2 alpha2, RowState& s, bin_t* bin,
                                             int wG, int valid, bool write, uint64_t pol, int c, int pos) {
  float2 acc = s.carry;
#pragma unroll
  for (int sg = 0; sg < kN / 16; ++sg) {
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const int c0 = sg * 16 + 2 * p;
      const float2 x = make_float2(__uint_as_float(r[sg][2 * p]), __uint_as_float(r[sg][2 * p + 1]));
      const float2 t = __ffma2_rn(x, alpha2, s.negR);
      float2 e = make_float2(ex2(t.x), ex2(t.y));
      if (MASK) {
        e.x = (c0 < valid) ? e.x : 0.f;
        e.y = (c0 + 1 < valid) ? e.y : 0.f;
      }
      if (pos + 1 == c) {                         // a chunk ends at the pair's first column
        const float bsum = (acc.x + acc.y) + e.x;
        if (write) st_keep(bin, bsum, pol);
        bin += wG;
        s.l += bsum;
        acc = make_float2(0.f, e.y);
        pos = 1;
      } else if (pos + 2 == c) {                  // a chunk ends at the pair's second column
        acc = __fadd2_rn(acc, e);
        const float bsum = acc.x + acc.y;
        if (write) st_keep(bin, bsum, pol);
        bin += wG;
        s.l += bsum;
        acc = make_float2(0.f, 0.f);
        pos = 0;
      } else {
        acc = __fadd2_rn(acc, e);
        pos += 2;
      }
    }
  }
  s.carry = acc;
}

// One tile of kN columns: compile-time chunk sizes take the pipelined segments;
// a chunk size known only at run time loads the whole row segment from TMEM
// first (kN/16 x16 loads, one wait) and counts its chunk ends.
template <int C, int PH, bool MASK, bool STORE>
__device__ __forceinline__ void tile_phase(uint32_t taddr, float2 alpha, RowState& s, bin_t* bin, int wG, int valid,
                                           bool write, uint64_t pol, int c, int ph) {
  if constexpr (C > 0) {
    uint32_t ra[16], rb[16];
    tmem_ld16(taddr, ra);
    tmem_wait16(ra);
    tile_segs_pipe<C, PH, 0, MASK, STORE>(taddr, ra, rb, alpha, s, bin, wG, valid, write, pol);
  } else {
    uint32_t r[kN / 16][16];
#pragma unroll
    for (int sg = 0; sg < kN / 16; ++sg) tmem_ld16(taddr + 16 * sg, r[sg]);
#pragma unroll
    for (int sg = 0; sg < kN / 16; ++sg) tmem_wait16(r[sg]);
    tile_cols_rt<MASK>(r, alpha, s, bin, wG, valid, write, pol, c, ph);
  }
}

// C > 0: the tile phases ph = (t * kN) mod C are the multiples of gcd(kN, C)
// below C, each a compile-time instance; C = 0 (chunk size c known at run time)
// passes the phase on.  STORE = false forms the row sums only (no bins).
template <int C, bool STORE, int PH = 0>
__device__ __forceinline__ void tile_dispatch(int ph, bool mask, uint32_t taddr, float2 alpha, RowState& s, bin_t* bin,
                                              int wG, int valid, bool write, uint64_t pol, int c) {
  if constexpr (C == 0) {
    if (mask)
      tile_phase<0, 0, true, STORE>(taddr, alpha, s, bin, wG, valid, write, pol, c, ph);
    else
      tile_phase<0, 0, false, STORE>(taddr, alpha, s, bin, wG, valid, write, pol, c, ph);
  } else if constexpr (PH < C) {
    if (ph == PH) {
      if (mask)
        tile_phase<C, PH, true, STORE>(taddr, alpha, s, bin, wG, valid, write, pol, c, ph);
      else
        tile_phase<C, PH, false, STORE>(taddr, alpha, s, bin, wG, valid, write, pol, c, ph);
    } else {
      tile_dispatch<C, STORE, PH + gcd_c(kN, C)>(ph, mask, taddr, alpha, s, bin, wG, valid, write, pol, c);
    }
  }
}

// Token-level chunks, second pass: the row's base-2 log-sum-exp L is known, so
// 2^(s * alpha - L) is the key's softmax probability in this row.  Each 16-column
// segment is summed over the warp's 32 rows by a transpose reduction (fin.cuh,
// warp_sum_each: lanes 2j and 2j + 1 end with column j's sum) and the even lanes
// store the warp's 16 column sums to `out` (the warp's partial array at the
// tile's column 0).  Padding rows carry L = +inf and add zeros.
template <int SEG, bool MASK>
__device__ __forceinline__ void direct_segs(uint32_t taddr, uint32_t (&ra)[16], uint32_t (&rb)[16], float2 alpha2,
                                            float2 negL, float* out, int valid, int lane) {
  if constexpr (SEG < kN / 16) {
    if constexpr (SEG + 1 < kN / 16) tmem_ld16(taddr + 16 * (SEG + 1), rb);
    float v[16];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const int c0 = SEG * 16 + 2 * p;
      const float2 x = make_float2(__uint_as_float(ra[2 * p]), __uint_as_float(ra[2 * p + 1]));
      const float2 t = __ffma2_rn(x, alpha2, negL);
      v[2 * p] = ex2(t.x);
      v[2 * p + 1] = ex2(t.y);
      if (MASK) {
        v[2 * p] = (c0 < valid) ? v[2 * p] : 0.f;
        v[2 * p + 1] = (c0 + 1 < valid) ? v[2 * p + 1] : 0.f;
      }
    }
    const int col = SEG * 16 + warp_sum_each<16>(v, lane);
    if (!(lane & 1) && (!MASK || col < valid)) out[col] = v[0];
    if constexpr (SEG + 1 < kN / 16) {
      tmem_wait16(rb);
      direct_segs<SEG + 1, MASK>(taddr, rb, ra, alpha2, negL, out, valid, lane);
    }
  }
}

// Row maximum of the first `valid` columns of a tile (raw dot products).
__device__ __forceinline__ float tile_max(uint32_t taddr, int valid) {
  float m = -INFINITY;
  uint32_t r[16];
#pragma unroll
  for (int sg = 0; sg < kN / 16; ++sg) {
    tmem_ld16(taddr + 16 * sg, r);
    tmem_wait16(r);
#pragma unroll
    for (int i = 0; i < 16; ++i) m = (16 * sg + i < valid) ? fmaxf(m, __uint_as_float(r[i])) : m;
  }
  return m;
}

// The 128 window rows of an item's M tile into shared memory (two 64-element
// panels, 128-byte swizzle), completing on bar.
__device__ __forceinline__ void load_q(const TcMaps& maps, const TcGeom& g, const Item& it, uint32_t sq, uint32_t bar) {
  mbar_expect_tx(bar, kQBytes);
  if (g.q_direct) {
    const CUtensorMap* qm = &maps.q[it.grp];
    const int hq0 = it.h * g.G + it.mt * g.qm;
    tma_load_4d(sq, qm, bar, 0, 0, hq0, it.b >> g.qshift);
    tma_load_4d(sq + kPanelQ, qm, bar, 64, 0, hq0, it.b >> g.qshift);
  } else {
    tma_load_2d(sq, &maps.q[0], bar, 0, it.key * 128);
    tma_load_2d(sq + kPanelQ, &maps.q[0], bar, 64, it.key * 128);
  }
}

// ---------------------------------------------------------------- the kernel
// WG > 0: the window rows per KV head are known at compile time (the common
// shapes), so each bin store of the softmax takes its address as base plus an
// immediate; WG = 0 reads them from the geometry.
// MODE 0: bins and (R, l) pairs (single pass).  Token-level chunks (C = 1) take
// two passes instead: MODE 1 writes only the (R, l) pairs, from which the
// log-sum-exp kernel forms each row's lse; MODE 2 reads lse and writes each key's
// probability summed over the rows of a warp (one partial array per warp of
// window rows, summed by sum_partials_kernel), so no bins are written or read.
template <int C, bool CAUSAL, int WG, int MODE = 0>
__global__ void __launch_bounds__(kThreads, 2)
score_tc_kernel(const __grid_constant__ TcMaps maps, TcGeom g, const __grid_constant__ SeqTable st,
                float* __restrict__ rl, bin_t* __restrict__ bins, int32_t* __restrict__ err,
                int32_t* __restrict__ sched, const float* __restrict__ lse_rows) {
  static_assert(MODE == 0 || (C == 1 && !CAUSAL), "two passes: token-level chunks without the causal window");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (smem_u32(smem_raw) & 1023u) {                         // swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicCAS(err, 0, (int)kDevMisalignedSmem);
    return;
  }
  uint8_t* sQ = smem;                                          // kStagesQ x 32 KB
  uint8_t* sK = smem + kStagesQ * kQBytes;                     // kStagesK x 20 KB
  uint64_t* bars = (uint64_t*)(sK + kStagesK * kKBytes);
  uint64_t* q_full = bars;                                     // [kStagesQ]
  uint64_t* q_empty = bars + kStagesQ;                         // [kStagesQ]
  uint64_t* k_full = bars + 2 * kStagesQ;                      // [kStagesK]
  uint64_t* k_empty = k_full + kStagesK;                       // [kStagesK]
  uint64_t* t_full = k_empty + kStagesK;                       // [kStagesT]
  uint64_t* t_empty = t_full + kStagesT;                       // [kStagesT]
  uint64_t* drained = t_empty + kStagesT;                      // [1] all MMAs done (teardown after a give-up)
  uint64_t* item_full = drained + 1;                           // [kItemRing]
  uint64_t* item_empty = item_full + kItemRing;                // [kItemRing]
  uint32_t* tmem_slot = (uint32_t*)(item_empty + kItemRing);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  volatile int* s_items = abort_flag + 1;                      // [kItemRing] claimed item (-1: none left)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStagesQ; ++i) { mbar_init(smem_u32(&q_full[i]), 1); mbar_init(smem_u32(&q_empty[i]), 1); }
    for (int i = 0; i < kStagesK; ++i) { mbar_init(smem_u32(&k_full[i]), 1); mbar_init(smem_u32(&k_empty[i]), 1); }
    for (int i = 0; i < kStagesT; ++i) { mbar_init(smem_u32(&t_full[i]), 1); mbar_init(smem_u32(&t_empty[i]), 128); }
    mbar_init(smem_u32(drained), 1);
    // an item is released by the MMA issuer and one lane of each softmax warp
    for (int i = 0; i < kItemRing; ++i) { mbar_init(smem_u32(&item_full[i]), 1); mbar_init(smem_u32(&item_empty[i]), 5); }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&maps.q[0]) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&maps.k[0]) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Ctl ctl{err, abort_flag, g.timeout};
  // copies issued by the producer (key tiles, window-row tiles): after a give-up
  // the teardown waits for the last phase armed on each of their barriers
  uint32_t kc = 0, qc = 0;
  const int cc = C > 0 ? C : g.c;                      // chunk size

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      pdl_wait();                                      // the packed window rows come from the previous launch
      int qkey = -1;                                   // (group, sequence, head, M tile) of the loaded Q
      // keys: normal priority, since the CTAs of the other M tiles of the same
      // (unit, head) read each key tile too (evict-first cost re-reads from HBM)
      const uint64_t kpol = policy_evict_normal();
      bool ok = true;
      for (uint32_t n = 0; ok && !*abort_flag; ++n) {
        // claim the next item of the launch and pass it on; -1 ends every role's loop
        const int slot = n % kItemRing;
        if (!wait_bar(ctl, smem_u32(&item_empty[slot]), ((n / kItemRing) & 1) ^ 1, kDevTimeoutTmaProducer)) break;
        int item = atomicAdd(&sched[0], 1);
        if (item >= g.n_items) item = -1;
        s_items[slot] = item;
        mbar_arrive(smem_u32(&item_full[slot]));
        if (item < 0) break;
        const Item it = decode_item(g, st, item);
        const CUtensorMap* kmap = &maps.k[it.grp];
        // A new window-row tile is loaded only after the first K tiles of the item
        // are on their way: the MMAs of the previous item still need the old tile,
        // and its reload then overlaps the softmax of the previous item's last tiles.
        const int pre = it.key != qkey ? min(it.ntile, kStagesK) : 0;
        for (int t = 0; t < it.ntile && ok; ++t) {
          if (t == pre && it.key != qkey) {
            if (!wait_bar(ctl, smem_u32(&q_empty[0]), (qc & 1) ^ 1, kDevTimeoutTmaProducer)) { ok = false; break; }
            load_q(maps, g, it, smem_u32(sQ), smem_u32(&q_full[0]));
            ++qc;
            qkey = it.key;
          }
          const int ks = kc % kStagesK;
          if (!wait_bar(ctl, smem_u32(&k_empty[ks]), ((kc / kStagesK) & 1) ^ 1, kDevTimeoutTmaProducer)) {
            ok = false;
            break;
          }
          const uint32_t kbar = smem_u32(&k_full[ks]);
          mbar_expect_tx(kbar, kKBytes);
          const int tok = (int)(it.tok0 + t * kN);
          tma_load_3d_hint(smem_u32(sK + ks * kKBytes), kmap, kbar, 0, it.h, tok, kpol);
          tma_load_3d_hint(smem_u32(sK + ks * kKBytes + kPanelK), kmap, kbar, 64, it.h, tok, kpol);
          ++kc;
        }
        if (ok && it.key != qkey) {          // an item shorter than the prefetch: its Q comes last
          if (!wait_bar(ctl, smem_u32(&q_empty[0]), (qc & 1) ^ 1, kDevTimeoutTmaProducer)) break;
          load_q(maps, g, it, smem_u32(sQ), smem_u32(&q_full[0]));
          ++qc;
          qkey = it.key;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t kc = 0, qc = 0, tc = 0;                 // this warp's own counts of the same phases
      int qkey = -1;
      const uint64_t qdesc = sw128_desc(smem_u32(sQ));   // the window-row tile never moves
      for (uint32_t n = 0; !*abort_flag; ++n) {
        const int slot = n % kItemRing;
        if (!wait_bar(ctl, smem_u32(&item_full[slot]), (n / kItemRing) & 1, kDevTimeoutMma)) break;
        const int item = s_items[slot];
        mbar_arrive(smem_u32(&item_empty[slot]));
        if (item < 0) break;
        const Item it = decode_item(g, st, item);
        const int ntile = it.ntile;
        const int key = it.key;
        if (key != qkey) {
          // the shared-memory tile is refilled only after the MMAs that read it are done
          if (qkey >= 0) tc_commit(smem_u32(&q_empty[0]));
          if (!wait_bar(ctl, smem_u32(&q_full[0]), qc & 1, kDevTimeoutMma)) break;
          tc_fence_after();
          ++qc;
          qkey = key;
        }
        bool ok = true;
        for (int t = 0; t < ntile; ++t) {
          const int ks = kc % kStagesK, ts = tc % kStagesT;
          if (!wait_bar(ctl, smem_u32(&k_full[ks]), (kc / kStagesK) & 1, kDevTimeoutMma) ||
              !wait_bar(ctl, smem_u32(&t_empty[ts]), ((tc / kStagesT) & 1) ^ 1, kDevTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t kdesc = sw128_desc(smem_u32(sK + ks * kKBytes));
          const uint32_t d = tmem + ts * kN;
          // step kk reads 16 bf16 (32 B) of every row: panel kk / 4, offset 32 (kk % 4) inside the
          // swizzle atom; the descriptors' start-address fields (16-byte units) advance by that
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = (kk & 3) * 32;
            tc_mma_ss(d, qdesc + (((kk >> 2) * kPanelQ + off) >> 4), kdesc + (((kk >> 2) * kPanelK + off) >> 4),
                      kk > 0 ? 1u : 0u);
          }
          tc_commit(smem_u32(&k_empty[ks]));
          tc_commit(smem_u32(&t_full[ts]));
          ++kc;
          ++tc;
        }
        if (!ok) break;
      }
    }
  } else {
    // ------------------------------------------------ softmax: one window row per thread
    // warps 2..5 cover the four TMEM lane groups (a warp reads lanes 32*(warp%4)..+31)
    const int lg = warp & 3;
    const int rloc = lg * 32 + lane;
    const uint64_t bpol = policy_evict_last();       // bins are read back by the finalisation
    pdl_wait();                                      // previous kernel of the stream done (and its writes visible)
    const uint32_t lane_base = tmem + ((uint32_t)(lg * 32) << 16);
    uint32_t tc = 0;
    for (uint32_t n = 0; !*abort_flag; ++n) {
      const int slot = n % kItemRing;
      if (!wait_bar(ctl, smem_u32(&item_full[slot]), (n / kItemRing) & 1, kDevTimeoutEpilogue)) break;
      const int item = s_items[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&item_empty[slot]));
      if (item < 0) break;
      const Item it = decode_item(g, st, item);
      const int nk = it.nk, ntile = it.ntile;
      const int row = it.mt * 128 + rloc;
      const int wg = WG > 0 ? WG : g.wG;                            // bin stride between chunks
      const bool warp_live = it.mt * 128 + lg * 32 < g.wG;         // whole warp of padding rows: no work
      if constexpr (MODE == 2) {
        const float2 alpha2 = make_float2(g.alpha, g.alpha);
        const float L = row < g.wG ? lse_rows[(int64_t)it.grp * (g.slot_bytes / 4) +
                                              ((int64_t)it.b * g.Hkv + it.h) * g.wG + row]
                                   : INFINITY;
        const float2 negL = make_float2(-L, -L);
        // this warp's partial array: warp p = 4 mt + lane quarter of the head's window rows
        float* part = (float*)((char*)bins + it.grp * g.slot_bytes) +
                      ((int64_t)(it.mt * 4 + lg) * g.Hkv + it.h) * st.cu[st.B] + it.tok0;
        bool ok = true;
        for (int t = 0; t < ntile; ++t) {
          const int ts = tc % kStagesT;
          if (!wait_bar(ctl, smem_u32(&t_full[ts]), (tc / kStagesT) & 1, kDevTimeoutEpilogue)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (warp_live) {
            const uint32_t taddr = lane_base + ts * kN;
            const int valid = min(kN, nk - t * kN);
            uint32_t ra[16], rb[16];
            tmem_ld16(taddr, ra);
            tmem_wait16(ra);
            if (valid < kN)
              direct_segs<0, true>(taddr, ra, rb, alpha2, negL, part + t * kN, valid, lane);
            else
              direct_segs<0, false>(taddr, ra, rb, alpha2, negL, part + t * kN, valid, lane);
          }
          tc_fence_before();
          mbar_arrive(smem_u32(&t_empty[ts]));
          ++tc;
        }
        if (!ok) break;
        continue;
      }
      // rows that own bins; with a compile-time w*G that is a multiple of 32 every row of a live warp
      // does, which lets the bin stores go without a branch each
      const bool write = (WG > 0 && WG % 32 == 0) ? warp_live : row < g.wG;
      bin_t* ubins = (bin_t*)((char*)bins + it.grp * g.slot_bytes) + (size_t)it.unit * g.cpu * g.wG + row;
      float* url = (float*)((char*)rl + it.grp * g.slot_bytes) + (size_t)it.unit * 2 * g.wG + row;
      RowState s{make_float2(0.f, 0.f), make_float2(0.f, 0.f), 0.f};
      const float2 alpha2 = make_float2(g.alpha, g.alpha);
      // causal window: packed position of the window's first query (T - w in the sequence)
      const int64_t causal_from = CAUSAL ? (int64_t)st.cu[it.b + 1] - g.w : 0;
      float R = 0.f;
      bool ok = true;
      for (int t = 0; t < ntile; ++t) {
        const int ts = tc % kStagesT;
        if (!wait_bar(ctl, smem_u32(&t_full[ts]), (tc / kStagesT) & 1, kDevTimeoutEpilogue)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (warp_live) {
          const uint32_t taddr = lane_base + ts * kN;
          int valid = min(kN, nk - t * kN);
          bool mask = valid < kN;
          if (CAUSAL && it.tok0 + t * kN + kN > causal_from) {
            // a tile reaching the window: the row's window query sees keys up to
            // T - w + (row mod w), a per-thread limit (the TMEM loads stay warp-wide)
            const int last = causal_from + row % g.w - (int)(it.tok0 + t * kN);
            valid = max(min(valid, last + 1), 0);
            mask = __any_sync(0xffffffffu, valid < kN);
          }
          if (t == 0) {
            R = tile_max(taddr, valid) * g.alpha + kBinShift;      // shifted reference (bin scale)
            s.negR = make_float2(-R, -R);
          }
          const int ph = (t * kN) % cc;
          const int q = (t * kN) / cc;
          const RowState before = s;
          tile_dispatch<C, MODE == 0>(ph, mask, taddr, alpha2, s, ubins + (size_t)q * wg, wg, valid, write, bpol, cc);
          // every bin is at most the row sum: one test per tile catches any value
          // that outgrew the reference (and inf / NaN)
          const bool over = !(s.l <= kBig);
          if (__any_sync(0xffffffffu, over)) {
            // those rows move their reference to this tile's maximum, rescale what
            // they already hold and redo the tile (the whole warp takes part because
            // the TMEM loads are warp-collective)
            const float tm = tile_max(taddr, valid) * g.alpha + kBinShift;
            const float R2 = over ? fmaxf(R, tm) : R;
            const float f = ex2(R - R2);
            if (MODE == 0 && over && write)
              for (int ch = 0; ch < q; ++ch)
                ubins[(size_t)ch * g.wG] = bin_encode(bin_decode(ubins[(size_t)ch * g.wG]) * f);
            s = before;
            s.l *= f;
            s.carry = make_float2(s.carry.x * f, s.carry.y * f);
            R = R2;
            s.negR = make_float2(-R2, -R2);
            tile_dispatch<C, MODE == 0>(ph, mask, taddr, alpha2, s, ubins + (size_t)q * wg, wg, valid, write, bpol, cc);
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&t_empty[ts]));
        ++tc;
      }
      if (!ok) break;
      if (warp_live && write) {
        // the item ended inside a chunk (last, partial chunk of the sequence)
        if (MODE == 0 && (ntile * kN) % cc != 0) {
          const float cs = s.carry.x + s.carry.y;
          const int ch = (ntile * kN) / cc;
          if (ch < g.cpu) ubins[(size_t)ch * g.wG] = bin_encode(cs);
          s.l += cs;
        }
        url[0] = R;
        url[g.wG] = s.l;
      }
    }
  }

  // ------------------------------------------------ teardown
  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    // The last CTA to finish (every producer has stopped claiming by then) sets
    // the item counter back to zero for the next launch on this workspace.
    __threadfence();
    if (atomicAdd(&sched[1], 1) == (int)gridDim.x - 1) {
      atomicExch(&sched[0], 0);
      atomicExch(&sched[1], 0);
    }
  }
  if (*abort_flag) {
    // A role gave up: copies and MMAs this CTA started may still be in flight, and
    // they must land before its shared memory and TMEM are released.  The producer
    // waits for the last phase it armed on every key stage and on the window-row
    // stage; the MMA issuer commits everything it issued to one more barrier and
    // waits for it.  Only if one of those bounded waits runs out does the CTA fall
    // back to a fixed pause.
    bool landed = true;
    if (warp == 0 && lane == 0) {
      for (uint32_t i = kc > kStagesK ? kc - kStagesK : 0; i < kc; ++i)
        landed &= drain_phase(smem_u32(&k_full[i % kStagesK]), (i / kStagesK) & 1, kDrainCycles);
      if (qc > 0) landed &= drain_phase(smem_u32(&q_full[0]), (qc - 1) & 1, kDrainCycles);
    }
    if (warp == 1 && lane == 0) {
      tc_commit(smem_u32(drained));
      landed &= drain_phase(smem_u32(drained), 0, kDrainCycles);
    }
    if (!landed) {
      const long long t0 = clock64();
      while (clock64() - t0 < kDrainCycles) {
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

// Packed window rows: qp[((b*Hkv + h)*MT + mt)*128 + r][e] = Q_w[b, r % w, h*G + r / w, e] for
// rows r < w*G of the group, zero for the padding rows up to MT*128.  blockIdx.y
// selects one of up to kMaxPackLayers layers (their packed tiles follow each other).
constexpr int kMaxPackLayers = 64;
struct PackArgs {
  int32_t n;
  const __nv_bfloat16* q[kMaxPackLayers];
};

__global__ void pack_q_kernel(const __grid_constant__ PackArgs pa, ScoreGeom g, int MT, int B,
                              __nv_bfloat16* __restrict__ qp_base, int64_t layer_elems) {
  const __nv_bfloat16* q = pa.q[blockIdx.y];
  __nv_bfloat16* qp = qp_base + blockIdx.y * layer_elems;
  pdl_wait();
  const int rows_per_head = MT * 128;
  const int64_t total_vec = (int64_t)B * g.Hkv * rows_per_head * (kD / 8);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total_vec; i += (int64_t)gridDim.x * blockDim.x) {
    const int vi = (int)(i % (kD / 8));
    const int64_t row = i / (kD / 8);
    const int r = (int)(row % rows_per_head);
    const int64_t bh = row / rows_per_head;
    const int h = (int)(bh % g.Hkv), b = (int)(bh / g.Hkv);
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r < g.wG) {
      const int gm = r / g.w, qi = r % g.w;
      val = *(const uint4*)(q + (int64_t)(b >> g.pair) * g.q_stride_b + (int64_t)qi * g.q_stride_w +
                            (int64_t)(h * g.G + gm) * g.q_stride_h + vi * 8);
    }
    *(uint4*)(qp + row * kD + vi * 8) = val;
  }
  pdl_trigger();
}

// Failure-path self test: one thread starts a real asynchronous copy (64 bytes
// of the workspace header, bytes 128..191, into shared memory by the bulk-copy
// engine), then waits, through the same bounded wait as the scoring kernel's
// roles, on an mbarrier phase that nothing completes.  The wait runs out after
// `timeout` clock64 cycles, records kDevTimeoutSelftest in the workspace error
// word and raises the CTA abort flag; the thread then drains the copy the way
// the scoring kernel's teardown does (a bounded wait on the copy's own barrier
// phase) and writes what landed to header bytes 64..127, so that a caller can
// see that the drain waited for the copy before the kernel returned.
__global__ void wait_selftest_kernel(int32_t* err, long long timeout) {
  __shared__ uint64_t bar;
  __shared__ uint64_t copied;
  __shared__ int abort_flag;
  __shared__ __align__(16) uint8_t buf[64];
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);                 // one arrival expected, none made
    mbar_init(smem_u32(&copied), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint8_t* src = reinterpret_cast<const uint8_t*>(err) + 128;
    mbar_expect_tx(smem_u32(&copied), 64);
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 64, [%2];"
        ::"r"(smem_u32(buf)), "l"((uint64_t)src), "r"(smem_u32(&copied)) : "memory");
    const Ctl ctl{err, (volatile int*)&abort_flag, timeout};
    if (wait_bar(ctl, smem_u32(&bar), 0, kDevTimeoutSelftest)) atomicExch(err, 0x7FFFFFFF);   // must not happen
    if (drain_phase(smem_u32(&copied), 0, kDrainCycles)) {
      uint8_t* dst = reinterpret_cast<uint8_t*>(err) + 64;
      for (int i = 0; i < 64; ++i) dst[i] = buf[i];
    }
  }
}

// ---------------------------------------------------------------- host side
using EncodeFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = (EncodeFn)p;
  });
  return fn;
}

struct DeviceInfo {
  int sms = 0;
  bool attr_set[64] = {};                       // per kernel instance (launch_c's slot)
};

DeviceInfo& device_info(int dev) {
  static DeviceInfo info[64];
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& d = info[dev & 63];
  if (d.sms == 0) cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  return d;
}

template <int C, bool CAUSAL, int WG, int MODE = 0>
cudaError_t launch_c(const TcGeom& tg, const TcMaps& maps, const SeqTable& st, float* rl, bin_t* bins, int32_t* err,
                     int slot, cudaStream_t s, const float* lse = nullptr) {
  int32_t* sched = err + kSchedWord;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  DeviceInfo& di = device_info(dev);
  if (!di.attr_set[slot]) {
    e = cudaFuncSetAttribute(score_tc_kernel<C, CAUSAL, WG, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    di.attr_set[slot] = true;
  }
  // Two CTAs per SM; each claims items from the counter until none are left, so
  // a CTA that drew short items (the last unit of a sequence) takes more.
  const int grid = std::min(tg.n_items, 2 * di.sms);
  return launch_pdl(score_tc_kernel<C, CAUSAL, WG, MODE>, dim3(grid), dim3(kThreads), (size_t)kSmemBytes, s, maps, tg,
                    st, rl, bins, err, sched, lse);
}

// Instances per chunk size: the causal window (any w*G), and without it w*G of
// 128, 256 and 448 at compile time (LLaMA / Mistral / Qwen-shaped GQA groups
// with 32- and 64-query windows) or any other w*G at run time.  `slot` numbers
// the chunk size's five instances for the one-time shared-memory attribute.
template <int C>
cudaError_t launch_causal(bool causal, const TcGeom& tg, const TcMaps& maps, const SeqTable& st, float* rl,
                          bin_t* bins, int32_t* err, int slot, cudaStream_t s) {
  if (causal) return launch_c<C, true, 0>(tg, maps, st, rl, bins, err, 5 * slot + 1, s);
  switch (tg.wG) {
    case 128: return launch_c<C, false, 128>(tg, maps, st, rl, bins, err, 5 * slot + 2, s);
    case 256: return launch_c<C, false, 256>(tg, maps, st, rl, bins, err, 5 * slot + 3, s);
    case 448: return launch_c<C, false, 448>(tg, maps, st, rl, bins, err, 5 * slot + 4, s);
    default: return launch_c<C, false, 0>(tg, maps, st, rl, bins, err, 5 * slot, s);
  }
}

// Chunk sizes without an instance of their own (C = 0: c read at run time): the
// causal window or any w*G.
template <int C>
cudaError_t launch_any_wg(bool causal, const TcGeom& tg, const TcMaps& maps, const SeqTable& st, float* rl,
                          bin_t* bins, int32_t* err, int slot, cudaStream_t s) {
  if (causal) return launch_c<C, true, 0>(tg, maps, st, rl, bins, err, 5 * slot + 1, s);
  return launch_c<C, false, 0>(tg, maps, st, rl, bins, err, 5 * slot, s);
}

// The two passes of token-level chunks (MODE 1, MODE 2) with the same w*G
// instances; slots 55 .. 62 of the one-time shared-memory attribute.
template <int MODE>
cudaError_t launch_two_pass(const TcGeom& tg, const TcMaps& maps, const SeqTable& st, float* rl, bin_t* bins,
                            int32_t* err, const float* lse, cudaStream_t s) {
  const int slot = 55 + 4 * (MODE - 1);
  switch (tg.wG) {
    case 128: return launch_c<1, false, 128, MODE>(tg, maps, st, rl, bins, err, slot + 1, s, lse);
    case 256: return launch_c<1, false, 256, MODE>(tg, maps, st, rl, bins, err, slot + 2, s, lse);
    case 448: return launch_c<1, false, 448, MODE>(tg, maps, st, rl, bins, err, slot + 3, s, lse);
    default: return launch_c<1, false, 0, MODE>(tg, maps, st, rl, bins, err, slot, s, lse);
  }
}

int lcm_i(int a, int b) { return a / gcd_c(a, b) * b; }

// Largest chunk size the tensor-core path takes: its units are whole tiles and
// whole chunks, lcm(80, c) keys at least.
constexpr int kMaxTcChunk = 4096;

}  // namespace tc

void tc_plan(Plan& pl) {
  pl.use_tc = 0;
  pl.tc_mt = 0;
  pl.tc_base_chunks = 0;
  // bf16 keys of head dimension 128 and any chunk size up to kMaxTcChunk (larger
  // chunks would make a whole-tile unit very long); the rest runs the SIMT kernel
  if (!(pl.elt == 2 && pl.d == tc::kD && pl.wG > 0 && pl.c >= 1 && pl.c <= tc::kMaxTcChunk)) return;
  // Units are whole tiles and whole chunks: multiples of lcm(80, c) keys.  The
  // multiplier is chosen by the planner (balance over the persistent grid).
  pl.use_tc = 1;
  pl.tc_mt = (pl.wG + 127) / 128;
  pl.tc_base_chunks = tc::lcm_i(tc::kN, pl.c) / pl.c;
  pl.tc_tile_n = tc::kN;
  pl.cpu = pl.tc_base_chunks * std::max(1, 640 / tc::lcm_i(tc::kN, pl.c));
}

cudaError_t launch_pack_q(const Plan& pl, const ScoreGeom& g, const void* const* q_layers, int n_layers,
                          void* qpack, cudaStream_t s) {
  const int MT = pl.tc_mt;
  const int64_t layer_elems = (int64_t)pl.B * pl.Hkv * MT * 128 * tc::kD;
  for (int l0 = 0; l0 < n_layers; l0 += tc::kMaxPackLayers) {
    tc::PackArgs pa;
    pa.n = std::min(tc::kMaxPackLayers, n_layers - l0);
    for (int i = 0; i < pa.n; ++i) pa.q[i] = (const __nv_bfloat16*)q_layers[l0 + i];
    const int64_t total_vec = layer_elems / 8;
    dim3 grid((unsigned)std::min<int64_t>((total_vec + 255) / 256, 2048), pa.n);
    cudaError_t e = launch_pdl(tc::pack_q_kernel, grid, dim3(256), 0, s, pa, g, MT, pl.B,
                               (__nv_bfloat16*)qpack + l0 * layer_elems, layer_elems);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

namespace tc {
// 4-D map over one layer's window queries Q_w [B, w, Hq, d] (see TcMaps).  The
// stride of an axis of extent 1 is never used and is then set to 16 bytes.
bool encode_q_direct(EncodeFn enc, CUtensorMap* map, const void* q, const Plan& pl, const ScoreGeom& g) {
  if (pl.w < 1 || 128 % pl.w != 0) return false;
  const int64_t ext[3] = {pl.w, (int64_t)pl.Hkv * pl.G, pl.B >> g.pair};   // window rows of B (or B / 2 caches)
  const int64_t st[3] = {g.q_stride_w, g.q_stride_h, g.q_stride_b};
  cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)ext[0], (cuuint64_t)ext[1], (cuuint64_t)ext[2]};
  cuuint64_t strides[3];
  for (int i = 0; i < 3; ++i) strides[i] = (cuuint64_t)(st[i] == 0 && ext[i] == 1 ? 16 : st[i] * 2);
  cuuint32_t box[4] = {64, (cuuint32_t)pl.w, (cuuint32_t)(128 / pl.w), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace tc

// Whether the scoring kernel can read the window rows from q itself (w divides
// 128 and the map encodes), so that no packing launch is needed.
bool tc_q_direct(const Plan& pl, const ScoreGeom& g, const void* q) {
  tc::EncodeFn enc = tc::encode_fn();
  CUtensorMap map;
  return pl.use_tc && pl.wG > 0 && pl.B > 0 && enc != nullptr && q != nullptr &&
         tc::encode_q_direct(enc, &map, q, pl, g);
}

// Scores n_groups layers (one per reuse group) in one persistent launch; group
// i reads keys k_groups[i] and writes the scratch slot at rl + i * slot_gs and
// bins + i * slot_gs (slot_gs in floats).  Window rows come from q_groups[i]
// itself when qpack is null (tc_q_direct said yes), otherwise packed back to
// back from qpack (launch_pack_q).  mode 1 and 2 are the two passes of token-level
// chunks (score_tc_kernel's MODE); mode 2 reads the rows' lse from lse + i * slot_gs
// and writes the partial arrays into the bins' place.
cudaError_t launch_score_tc(const Plan& pl, const ScoreGeom& g, const SeqTable& st, const void* const* q_groups,
                            const void* const* k_groups, int n_groups, int64_t slot_bytes, float* rl, bin_t* bins,
                            const void* qpack, int32_t* err, cudaStream_t s, int mode, const float* lse) {
  const bool direct = qpack == nullptr;
  tc::EncodeFn enc = tc::encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  const int MT = pl.tc_mt;
  const int T_total = st.cu[st.B];
  if (g.n_units == 0 || T_total == 0 || n_groups == 0) return cudaSuccess;
  const int64_t rows_pg = (int64_t)pl.B * pl.Hkv * MT * 128;
  for (int g0 = 0; g0 < n_groups; g0 += tc::kMaxGroups) {
    const int n = std::min(tc::kMaxGroups, n_groups - g0);
    static thread_local tc::TcMaps maps;
    if (direct) {
      for (int i = 0; i < n; ++i)
        if (!tc::encode_q_direct(enc, &maps.q[i], q_groups[g0 + i], pl, g)) return cudaErrorInvalidValue;
    } else {
      cuuint64_t dims[2] = {(cuuint64_t)tc::kD, (cuuint64_t)(rows_pg * n)};
      cuuint64_t strides[1] = {(cuuint64_t)tc::kD * 2};
      cuuint32_t box[2] = {64, 128};
      cuuint32_t es[2] = {1, 1};
      const void* qg = (const char*)qpack + g0 * rows_pg * tc::kD * 2;
      if (enc(&maps.q[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(qg), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
    for (int i = 0; i < n; ++i) {
      cuuint64_t dims[3] = {(cuuint64_t)tc::kD, (cuuint64_t)pl.Hkv, (cuuint64_t)T_total};
      cuuint64_t strides[2] = {(cuuint64_t)g.kv_stride_h * 2, (cuuint64_t)g.kv_stride_t * 2};
      cuuint32_t box[3] = {64, 1, tc::kN};
      cuuint32_t es[3] = {1, 1, 1};
      if (enc(&maps.k[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(k_groups[g0 + i]), dims, strides,
              box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
    tc::TcGeom tg = {};
    tg.B = pl.B;
    tg.Hkv = pl.Hkv;
    tg.wG = pl.wG;
    tg.MT = MT;
    tg.cpu = pl.cpu;
    tg.ku = pl.ku;
    tg.c = pl.c;
    tg.w = g.w;
    tg.G = pl.G;
    tg.q_direct = direct ? 1 : 0;
    tg.qm = direct ? 128 / pl.w : 0;
    tg.qshift = g.pair;
    tg.items_pg = g.n_units * MT;
    tg.n_items = tg.items_pg * n;
    tg.slot_bytes = slot_bytes;
    tg.alpha = g.alpha;
    tg.timeout = 4000000000LL;     // about two seconds of clock64 cycles per wait
    float* rlg = (float*)((char*)rl + g0 * slot_bytes);
    bin_t* bg = (bin_t*)((char*)bins + g0 * slot_bytes);
    if (mode == 1 || mode == 2) {
      const float* lg = lse ? (const float*)((const char*)lse + g0 * slot_bytes) : nullptr;
      const cudaError_t e = mode == 1 ? tc::launch_two_pass<1>(tg, maps, st, rlg, bg, err, lg, s)
                                      : tc::launch_two_pass<2>(tg, maps, st, rlg, bg, err, lg, s);
      if (e != cudaSuccess) return e;
      continue;
    }
    // compile-time instances (the chunk ends of every tile phase are constants) for
    // the common chunk sizes (the notes' ablation set 1, 3, 5, 10, 15, 20, 30 among
    // them); any other c >= 2 runs the C = 0 instance
    const bool causal = g.causal != 0;
    cudaError_t e = cudaErrorNotSupported;
    switch (pl.c) {
      case 1: e = tc::launch_causal<1>(causal, tg, maps, st, rlg, bg, err, 8, s); break;
      case 3: e = tc::launch_causal<3>(causal, tg, maps, st, rlg, bg, err, 0, s); break;
      case 4: e = tc::launch_causal<4>(causal, tg, maps, st, rlg, bg, err, 1, s); break;
      case 5: e = tc::launch_causal<5>(causal, tg, maps, st, rlg, bg, err, 2, s); break;
      case 8: e = tc::launch_causal<8>(causal, tg, maps, st, rlg, bg, err, 3, s); break;
      case 10: e = tc::launch_causal<10>(causal, tg, maps, st, rlg, bg, err, 4, s); break;
      case 16: e = tc::launch_causal<16>(causal, tg, maps, st, rlg, bg, err, 5, s); break;
      case 20: e = tc::launch_causal<20>(causal, tg, maps, st, rlg, bg, err, 6, s); break;
      case 30: e = tc::launch_causal<30>(causal, tg, maps, st, rlg, bg, err, 7, s); break;
      case 15: e = tc::launch_causal<15>(causal, tg, maps, st, rlg, bg, err, 10, s); break;
      default: e = tc::launch_any_wg<0>(causal, tg, maps, st, rlg, bg, err, 9, s); break;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

namespace tc {
// Token-level chunk scores from the second pass's partial arrays: the score of
// key j of (sequence b, KV head h) is the sum, in warp order, of the n_parts
// partial sums part[p][h][cu[b] + j] (one per warp of the head's window rows).
__global__ void sum_partials_kernel(ScoreGeom g, const __grid_constant__ SeqTable st, const float* __restrict__ part,
                                    int64_t slot_floats, int n_parts, float* __restrict__ scores) {
  const int bh = blockIdx.y;
  const int b = bh / g.Hkv, h = bh - b * g.Hkv;
  part += blockIdx.z * slot_floats;
  scores += blockIdx.z * g.scores_gs + (int64_t)bh * g.C_max;
  pdl_wait();
  const int T = st.cu[b + 1] - st.cu[b];
  const int64_t T_total = st.cu[st.B];
  const float* src = part + (int64_t)h * T_total + st.cu[b];
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < T; j += gridDim.x * blockDim.x) {
    float a = 0.f;
    for (int p = 0; p < n_parts; ++p) a += __ldcs(src + (int64_t)p * g.Hkv * T_total + j);
    scores[j] = a;
  }
  pdl_trigger();
}
}  // namespace tc

// Partial arrays of n_groups consecutive slots (at `part`, slot_bytes apart)
// into their token-level chunk scores.
cudaError_t launch_sum_partials(const Plan& pl, const ScoreGeom& g, const SeqTable& st, const float* part,
                                int64_t slot_bytes, float* scores, int n_groups, cudaStream_t s) {
  if (pl.B * pl.Hkv == 0 || n_groups == 0 || pl.C_max == 0) return cudaSuccess;
  const int n_parts = (pl.wG + 31) / 32;
  const dim3 grid((unsigned)std::min(64, (pl.C_max + 1023) / 1024), pl.B * pl.Hkv, n_groups);
  return launch_pdl(tc::sum_partials_kernel, grid, dim3(256), 0, s, g, st, part, slot_bytes / (int64_t)sizeof(float),
                    n_parts, scores);
}

cudaError_t launch_wait_selftest(int32_t* err, long long timeout, cudaStream_t s) {
  tc::wait_selftest_kernel<<<1, 32, 0, s>>>(err, timeout);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) g_launch_count.fetch_add(1, std::memory_order_relaxed);
  return e;
}

}  // namespace chunkkv
