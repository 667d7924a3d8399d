// pa_prefill_tc.cu -- chunked-prefill attention over the paged pool on the
// fifth-generation tensor cores (tcgen05 + tensor memory) of sm_103a.
//
// Pages: course README "Build an LLM Inference Engine From Scratch",
// curriculum row "Batching & Scheduling" (chunked prefill, FlashAttention) and
// the claims "chunked prefill produces a bit-identical KV cache" / "online
// softmax is exact"; "S20 - The Complete Engine", section "The conflicts"
// (prefill runs eagerly next to decode). A chunk of Lq queries at the end of a
// context of c tokens: query j sits at position c - Lq + j and (causal) sees
// keys 0 .. c - Lq + j, the earlier ones already in the cache.
//
// A prefill chunk gives each KV head (128/G) x G query rows that share every
// K/V tile: a real matrix product, so it runs on tcgen05 with accumulators in
// tensor memory. One CTA per SM, warp-specialised (11 warps):
//   warp 0    TMA producer for the query tiles (3-D tensor map over q; two
//             buffers, so the next piece's tile lands early) and for K, as
//             eight 16-key pool blocks per 128-key tile found through the
//             block table (ids fetched one tile ahead);
//   warp 10   TMA producer for V; K and V stages have their own full/empty
//             mbarriers, so a K stage refills as soon as its S is done;
//   warp 1    allocates 512 TMEM columns and, from one thread, issues the
//             MMAs: S = Q K^T into one of two S buffers (the next tile's S is
//             computed while softmax works on this one), then O_h += P_h V_h
//             for the two 64-key halves, with P read from tensor memory; each
//             finished group is signalled by tcgen05.commit on an mbarrier;
//   warps 2-9 softmax, two threads per query row, one per 64-key half, each
//             with its own running max, sum and O accumulator: read the S
//             half from TMEM, mask, exp2, write P (bf16 pairs) back over the S
//             columns just read; rescale O in TMEM only when a row maximum
//             grows by more than 2^8 (exact either way); at the end of a piece
//             the halves exchange (max, sum) through shared memory and write
//             the normalised row during the next tile.
// Work is a cut of the batch's flat (query tile, KV head, key tile) list at
// CTA granularity in which a segment start weighs as much as one key tile
// (PieceCut); pieces of a segment cut between CTAs are merged by
// prefill_tc_fixup_kernel. Beside a verify grid of the same call the grid
// keeps only its share of the SMs (overlap_split). Optional fp32 row output
// with a row map serves the cascade's shared-prefix half.
#include <cudaTypedefs.h>

#include "pa_device.cuh"
#include "pa_host.h"

namespace pa {
namespace {

constexpr int kRowsT = 128;                 // query rows per tile (MMA M)
constexpr int kKeysT = 128;                 // keys per tile (N of S, K of PV)
constexpr int kBlocksT = kKeysT / kBlock;   // pool blocks per key tile
constexpr int kHalfT = kRowsT * 128;        // one 64-column half of a 128-row bf16 operand
constexpr int kOpBytes = 2 * kHalfT;        // a 128 x 128 bf16 operand
constexpr int kOffQ = 0;                   // two query-tile buffers
constexpr int kOffKV = kOffQ + 2 * kOpBytes;  // stage s: K at kOffKV + s * 2 * kOpBytes, V after it
constexpr int kOffBar = kOffKV + 2 * 2 * kOpBytes;
constexpr int kNumBars = 20;
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
constexpr int kOffLx = kOffBar + 256;       // [2 pieces][2 halves][128 rows] x (m, l)
constexpr int kOffPlan = kOffLx + 2 * 2 * kRowsT * 8;
// a segment start weighs as much as one key tile in the cut between CTAs
// (measured: a CTA whose range starts many short segments spends about one
// tile's time more on each)
constexpr int kPieceCost4 = 4;
constexpr int kSoftmaxWarps = 8;            // warps 2-9, two per SM sub-partition
constexpr int kVWarp = 2 + kSoftmaxWarps;   // the V producer
constexpr int kThreadsT = 96 + kSoftmaxWarps * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;             // S/P buffers at columns 0 and 128; O halves at 256, 384
constexpr float kRescaleLog2 = 8.f;         // lazy O rescale threshold (log2 units)

enum : int {
  B_QFULL = 0, B_QFULL1, B_QEMPTY, B_QEMPTY1,
  B_KFULL, B_KFULL1, B_KEMPTY, B_KEMPTY1,
  B_VFULL, B_VFULL1, B_VEMPTY, B_VEMPTY1,
  B_SFULL, B_SFULL1, B_SFREE, B_SFREE1,
  B_PFULL, B_ODONE, B_LX, B_LX1
};

struct TcArgs {
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* cu_seqlens_q;
  uint16_t* out;
  float* lse;
  float scale_log2;
  int S, Hq, Hkv, G, QTb, max_blocks;
  int64_t num_blocks;
  int64_t num_q_tokens;
  int causal;
  int npairs_cap;
  int num_workers;
  // > 0: this grid runs beside the verify grid of the same call and keeps
  // overlap_split(...) of its split CTAs (one per SM); the others leave at once
  int split;
  int min_lq;
  float* part_o;    // [NW * 2][128 rows][128]
  float* part_lse;  // [NW * 2][128 rows]
  RowsOut rows;     // fp32 row output instead of out / lse (rows.o set)
  const int32_t* row_map;  // rows mode: query token i -> output token row_map[i]
};

// Output row (token * Hq + head) of query token qtok, head hd; -1 when the
// row map sends it outside the output (flagged, not written).
__device__ __forceinline__ int64_t out_row(const TcArgs& a, int64_t qtok, int hd) {
  if (!a.row_map) return qtok * a.Hq + hd;
  const int64_t t = a.row_map[qtok];
  if (t < 0 || t >= a.rows.tokens) {
    flag_error(PA_DEVERR_QLEN_RANGE);
    return -1;
  }
  return t * a.Hq + hd;
}

// ---------------------------------------------------------------------------
// tcgen05 / TMA wrappers
// ---------------------------------------------------------------------------

// Shared-memory matrix descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// kind::f16 instruction descriptor: fp32 accumulate, bf16 A and B, A K-major,
// B K-major (b_mn = 0) or MN-major (1).
__host__ __device__ constexpr uint32_t f16_idesc(int M, int N, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// A (M x K, K-major) read from tensor memory at column a_tmem, B from shared memory.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

#define PA_R32(x)                                                                            \
  "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]),       \
      "=r"(x[7]), "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]), \
      "=r"(x[14]), "=r"(x[15]), "=r"(x[16]), "=r"(x[17]), "=r"(x[18]), "=r"(x[19]),          \
      "=r"(x[20]), "=r"(x[21]), "=r"(x[22]), "=r"(x[23]), "=r"(x[24]), "=r"(x[25]),          \
      "=r"(x[26]), "=r"(x[27]), "=r"(x[28]), "=r"(x[29]), "=r"(x[30]), "=r"(x[31])
#define PA_W32(x)                                                                            \
  "r"(x[0]), "r"(x[1]), "r"(x[2]), "r"(x[3]), "r"(x[4]), "r"(x[5]), "r"(x[6]), "r"(x[7]),    \
      "r"(x[8]), "r"(x[9]), "r"(x[10]), "r"(x[11]), "r"(x[12]), "r"(x[13]), "r"(x[14]),      \
      "r"(x[15]), "r"(x[16]), "r"(x[17]), "r"(x[18]), "r"(x[19]), "r"(x[20]), "r"(x[21]),    \
      "r"(x[22]), "r"(x[23]), "r"(x[24]), "r"(x[25]), "r"(x[26]), "r"(x[27]), "r"(x[28]),    \
      "r"(x[29]), "r"(x[30]), "r"(x[31])
#define PA_REGS32                                                                         \
  "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22," \
  "%23,%24,%25,%26,%27,%28,%29,%30,%31}"

// 32 consecutive TMEM columns of this thread's lane (32x32b shape); the
// registers are valid after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 " PA_REGS32 ", [%32];"
               : PA_R32(v)
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&v)[32]) {
  // the registers are named as in/out operands so no use moves above the wait
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                 "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                 "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]),
                 "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]),
                 "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]),
                 "+r"(v[30]), "+r"(v[31])
               :
               : "memory");
}
// Orders later uses of v after an earlier tmem_wait_ld() (no instruction).
__device__ __forceinline__ void tmem_tie(uint32_t (&v)[32]) {
  asm volatile(""
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                 "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                 "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]),
                 "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]),
                 "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]),
                 "+r"(v[30]), "+r"(v[31]));
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  tmem_ld32_async(taddr, v);
  tmem_wait_ld(v);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,"
               "%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,"
               "%30,%31,%32};" ::"r"(taddr),
               PA_W32(v)
               : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void plan_inputs(const TcArgs& a, PlanInputs& in) {
  in.context_lens = a.context_lens;
  in.cu_seqlens_q = a.cu_seqlens_q;
  in.S = a.S;
  in.Hkv = a.Hkv;
  in.max_ctx = a.max_blocks * kBlock;
  in.qtile = a.QTb;
  in.causal = a.causal;
  in.npairs_cap = a.npairs_cap;
  in.num_q_rows = a.num_q_tokens;
  in.key_tile = kKeysT;
  in.min_lq = a.min_lq;
}

__device__ __forceinline__ void plan_view(unsigned char* base, const TcArgs& a, PlanSmem& P) {
  int* pm = reinterpret_cast<int*>(base);
  P.pair_off = pm;
  P.seq_pair = pm + (a.npairs_cap + 1);
  P.ctx = P.seq_pair + (a.S + 1);
  P.qstart = P.ctx + a.S;
}

// The worker starts of the piece-weighted cut, after the plan arrays.
__device__ __forceinline__ int* cut_view(unsigned char* base, const TcArgs& a) {
  return reinterpret_cast<int*>(base) + (a.npairs_cap + 1) + 3 * (a.S + 1);
}

// Two words for the SM split's reduction, after the cut (8-byte aligned).
__device__ __forceinline__ unsigned long long* split_view(unsigned char* base, const TcArgs& a) {
  const uintptr_t p = reinterpret_cast<uintptr_t>(cut_view(base, a) + a.num_workers + 1);
  return reinterpret_cast<unsigned long long*>((p + 7) & ~uintptr_t(7));
}

// The CTAs this call's prefill grid works with (all of them unless it runs
// beside the verify grid).
__device__ __forceinline__ int prefill_workers(const TcArgs& a, unsigned char* plan_base) {
  if (a.split <= 0) return a.num_workers;
  const int K = overlap_split(a.cu_seqlens_q, a.context_lens, a.S, a.Hkv, a.G, a.causal,
                              a.min_lq, a.max_blocks * kBlock, a.split,
                              split_view(plan_base, a));
  return min(a.num_workers, K);
}

__global__ void __launch_bounds__(kThreadsT, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmq,
                            const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv, const TcArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);
  const int S = a.S, Hkv = a.Hkv, G = a.G, QTb = a.QTb;
  auto bar = [&](int i) { return smem_addr(&bars[i]); };

  PlanSmem P;
  plan_view(smem + kOffPlan, a, P);
  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      const bool all = i == B_PFULL || i == B_LX || i == B_LX1;
      mbar_init(bar(i), all ? (uint32_t)(kSoftmaxWarps * 32) : 1u);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (tid == 32) {
    prefetch_tensormap(&tmq);
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  // launched as a programmatic dependent of the previous grid
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int max_workers = prefill_workers(a, smem + kOffPlan);
  // beside a verify grid: the CTAs past the split leave now, freeing their SMs
  if ((int)blockIdx.x >= max_workers) return;
  PlanInputs in;
  plan_inputs(a, in);
  build_plan(in, P, nullptr);  // ends with a CTA barrier
  const PieceCut cut = build_piece_cut(P, Hkv, max_workers, kPieceCost4, cut_view(smem + kOffPlan, a));
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int w = blockIdx.x;
  if (w >= cut.nw) return;  // the whole CTA is idle (uniform)
  const int R0 = cut.start(w), R1 = cut.start(w + 1);
  if (R0 >= R1) return;

  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto wait = [&](int b, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (!mbar_wait_bounded(bar(b), parity)) {
      *abort_flag = 1;
      return false;
    }
    return true;
  };

  if (warp == 0 || warp == kVWarp) {
    // ------------------------------------------------------------------ producers
    // warp 0 loads the query tiles and K, warp kVWarp loads V: each stage's K
    // is refilled as soon as its S is done, without queueing behind the V of
    // the previous tile (which waits for that tile's PV)
    const bool is_k = warp == 0;
    TilePos t = locate(P, S, Hkv, R0);
    auto nblocks_of = [&](const TilePos& tp) {
      const int nb_seq = (P.ctx[tp.s] + kBlock - 1) / kBlock;
      return min(kBlocksT, nb_seq - tp.b * kBlocksT);
    };
    auto fetch_ids = [&](const TilePos& tp) -> int {
      return lane < nblocks_of(tp)
                 ? a.block_tables[(size_t)tp.s * a.max_blocks + tp.b * kBlocksT + lane]
                 : 0;
    };
    const CUtensorMap* map = is_k ? &tmk : &tmv;
    const int b_full = is_k ? B_KFULL : B_VFULL, b_empty = is_k ? B_KEMPTY : B_VEMPTY;
    int ids = fetch_ids(t);
    int qn = 0;
    for (int idx = R0, i = 0; idx < R1; ++idx, ++i) {
      const bool first = (idx == R0) || (t.b == 0);
      if (is_k && first) {
        const int qs = qn & 1;
        if (qn >= 2 && !wait(B_QEMPTY + qs, (uint32_t)((qn >> 1) - 1) & 1u)) break;
        if (lane == 0) {
          const int z = P.qstart[t.s] + t.qt * QTb;  // first query token of the tile
          const uint32_t qd = smem_addr(smem + kOffQ + qs * kOpBytes);
          mbar_arrive_expect_tx(bar(B_QFULL + qs), kOpBytes);
          tma_load_3d(qd, &tmq, 0, t.h * G, z, bar(B_QFULL + qs));
          tma_load_3d(qd + kHalfT, &tmq, 64, t.h * G, z, bar(B_QFULL + qs));
        }
        ++qn;
      }
      const int st = i & 1;
      const int nb = nblocks_of(t);
      int my_id = ids;
      if (idx + 1 < R1) {  // block ids of the next tile, one tile ahead
        TilePos tn = t;
        advance(P, S, Hkv, tn);
        ids = fetch_ids(tn);
      }
      if (lane < nb && (my_id < 0 || (int64_t)my_id >= a.num_blocks)) {
        if (is_k) flag_error(PA_DEVERR_BLOCK_RANGE);
        my_id = 0;
      }
      const int y = (int)(((int64_t)my_id * Hkv + t.h) * kBlock);
      // the stage is free once the S (K) or the PV (V) of tile i-2 is done
      if (i >= 2 && !wait(b_empty + st, (uint32_t)((i >> 1) - 1) & 1u)) break;
      if (lane == 0) mbar_arrive_expect_tx(bar(b_full + st), (uint32_t)nb * (uint32_t)kTileBytes);
      __syncwarp();
      const uint32_t d = smem_addr(smem + kOffKV + st * 2 * kOpBytes + (is_k ? 0 : kOpBytes) +
                                   lane * (kBlock * 128));
      if (lane < nb) {
        tma_load_2d(d, map, 0, y, bar(b_full + st));
        tma_load_2d(d + kHalfT, map, 64, y, bar(b_full + st));
      }
      __syncwarp();
      if (idx + 1 < R1) advance(P, S, Hkv, t);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idS = f16_idesc(kRowsT, kKeysT, 0);
      const uint32_t idPV = f16_idesc(kRowsT, 128, 1);
      int qn = 0, qs = 0;  // query tiles seen; buffer of the current one
      auto issue_S = [&](int i, bool first) -> bool {
        if (first) {
          qs = qn & 1;
          if (!wait(B_QFULL + qs, (uint32_t)(qn >> 1) & 1u)) return false;
          ++qn;
        }
        const int st = i & 1;
        if (!wait(B_KFULL + st, (uint32_t)(i >> 1) & 1u)) return false;
        // the S/P buffer is free once the PV that read P of tile i-2 is done
        if (i >= 2 && !wait(B_SFREE + st, (uint32_t)((i >> 1) - 1) & 1u)) return false;
        tc_fence_after();
        const uint32_t sQ = smem_addr(smem + kOffQ + qs * kOpBytes);
        const uint32_t sK = smem_addr(smem + kOffKV + st * 2 * kOpBytes);
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // head_dim 128 = 8 steps of 16
          const uint32_t off = (uint32_t)(k >> 2) * kHalfT + (uint32_t)(k & 3) * 32u;
          tc_mma(tmem + (uint32_t)st * 128u, sw128_desc(sQ + off, 16, 1024),
                 sw128_desc(sK + off, 16, 1024), idS, k > 0);
        }
        tc_commit(bar(B_SFULL + st));
        tc_commit(bar(B_KEMPTY + st));
        return true;
      };
      TilePos t = locate(P, S, Hkv, R0);
      bool ok = issue_S(0, true);
      if (ok && (R0 + 1 >= R1 || t.b == t.nt - 1)) tc_commit(bar(B_QEMPTY + qs));
      for (int idx = R0, i = 0; ok && idx < R1; ++idx, ++i) {
        const bool first = (idx == R0) || (t.b == 0);
        if (idx + 1 < R1) {
          // the next tile's S first: the tensor core computes it during softmax
          TilePos tn = t;
          advance(P, S, Hkv, tn);
          if (!issue_S(i + 1, tn.b == 0)) {
            ok = false;
            break;
          }
          if (idx + 2 >= R1 || tn.b == tn.nt - 1) tc_commit(bar(B_QEMPTY + qs));
        }
        const int st = i & 1;
        if (!wait(B_PFULL, (uint32_t)i & 1u) || !wait(B_VFULL + st, (uint32_t)(i >> 1) & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sV = smem_addr(smem + kOffKV + st * 2 * kOpBytes + kOpBytes);
        // O_hf += P[:, keys of half hf] V[keys of half hf, :]: one accumulator per
        // key half; P (bf16 pairs) sits in columns st*128 + hf*64 .. +31 of TMEM
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc_mma_ts(tmem + kColO + (uint32_t)hf * 128u,
                      tmem + (uint32_t)st * 128u + (uint32_t)hf * 64u + (uint32_t)k * 8u,
                      sw128_desc(sV + (uint32_t)(hf * 4 + k) * 2048u, kHalfT, 1024), idPV,
                      (k > 0 || !first) ? 1u : 0u);
        tc_commit(bar(B_VEMPTY + st));
        tc_commit(bar(B_SFREE + st));
        tc_commit(bar(B_ODONE));
        if (idx + 1 < R1) advance(P, S, Hkv, t);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax
    // Thread (row r, half hf) owns keys hf*64 .. hf*64+63 of every tile of row r
    // with its own running maximum, sum and O accumulator; the two halves of a
    // row are merged once, at the end of a piece.
    const int q4 = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int r = q4 * 32 + lane;  // this thread's query row (= TMEM lane)
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const uint32_t tO = tmem + lane_base + kColO;
    float* lx = reinterpret_cast<float*>(smem + kOffLx);
    const float sc = a.scale_log2;
    TilePos t = locate(P, S, Hkv, R0);
    float m_ref = neg_inf(), l = 0.f;
    int lim = 0, c = 0, lq = 0, tok = 0, piece_b0 = 0, np = 0;
    bool valid = false, piece_first = true;
    // A finished piece's O stays in TMEM until the next tile's exponentials
    // are done (its last PV completes meanwhile); then it is written out.
    bool pend = false, pend_complete = false, pend_valid = false;
    int pend_np = 0;
    int64_t pend_orow = 0;
    size_t pend_slot = 0;
    float pend_m = 0.f, pend_l = 0.f;
    auto flush = [&]() -> bool {
      // merge the two key halves of the row: the partner's (m, l) from shared memory
      if (!wait(B_LX + (pend_np & 1), (uint32_t)(pend_np >> 1) & 1u)) return false;
      const float* other = lx + ((pend_np & 1) * 2 + (hf ^ 1)) * kRowsT * 2 + r * 2;
      const float m_o = other[0], l_o = other[1];
      const float M = fmaxf(pend_m, m_o);
      const float a_me = pend_m == neg_inf() ? 0.f : ex2(pend_m - M);
      const float a_o = m_o == neg_inf() ? 0.f : ex2(m_o - M);
      const float lt = pend_l * a_me + l_o * a_o;
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const float c0 = (hf == 0 ? a_me : a_o) * inv, c1 = (hf == 0 ? a_o : a_me) * inv;
      const float lse_v = lt > 0.f ? (M + lg2(lt)) * kLn2 : neg_inf();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int d0 = hf * 64 + cc * 32;  // output dims d0 .. d0+31
        uint32_t u0[32], u1[32];
        tmem_ld32_async(tO + (uint32_t)d0, u0);
        tmem_ld32_async(tO + 128u + (uint32_t)d0, u1);
        tmem_wait_ld(u0);
        tmem_tie(u1);
        float o[32];
#pragma unroll
        for (int j = 0; j < 32; ++j)
          o[j] = fmaf(__uint_as_float(u0[j]), c0, __uint_as_float(u1[j]) * c1);
        if (pend_complete && a.rows.o) {
          if (pend_valid) {
            float4* dst = reinterpret_cast<float4*>(
                a.rows.o + (pend_orow * a.rows.stride + a.rows.slot) * kHeadDim + d0);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
          }
        } else if (pend_complete) {
          if (pend_valid) {
            uint4* dst = reinterpret_cast<uint4*>(a.out + pend_orow * kHeadDim + d0);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(cvt_bf16x2(o[8 * q + 0], o[8 * q + 1]),
                                  cvt_bf16x2(o[8 * q + 2], o[8 * q + 3]),
                                  cvt_bf16x2(o[8 * q + 4], o[8 * q + 5]),
                                  cvt_bf16x2(o[8 * q + 6], o[8 * q + 7]));
          }
        } else {
          float4* dst =
              reinterpret_cast<float4*>(a.part_o + (pend_slot * kRowsT + r) * kHeadDim + d0);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        }
      }
      if (hf == 0) {
        if (pend_complete && a.rows.o) {
          if (pend_valid) a.rows.lse[pend_orow * a.rows.stride + a.rows.slot] = lse_v;
        } else if (pend_complete) {
          if (pend_valid && a.lse) a.lse[pend_orow] = lse_v;
        } else {
          a.part_lse[pend_slot * kRowsT + r] = lse_v;
        }
      }
      pend = false;
      return true;
    };
    int i = 0;
    for (int idx = R0; idx < R1; ++idx, ++i) {
      const bool first = (idx == R0) || (t.b == 0);
      const bool last = (idx == R1 - 1) || (t.b == t.nt - 1);
      if (first) {
        c = P.ctx[t.s];
        lq = P.qstart[t.s + 1] - P.qstart[t.s];
        tok = t.qt * QTb + r / G;
        valid = tok < lq;
        lim = valid ? (a.causal ? c - lq + tok + 1 : c) : 0;
        m_ref = neg_inf();
        l = 0.f;
        piece_b0 = t.b;
        piece_first = (idx == R0);
      }
      const int sb = i & 1;
      if (!wait(B_SFULL + sb, (uint32_t)(i >> 1) & 1u)) break;
      tc_fence_after();
      uint32_t v0[32], v1[32];
      const uint32_t tS = tmem + lane_base + (uint32_t)sb * 128u + (uint32_t)hf * 64u;
      tmem_ld32_async(tS, v0);
      tmem_ld32_async(tS + 32u, v1);
      tmem_wait_ld(v0);
      tmem_tie(v1);

      // scores in log2 units
      float2 x[32];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        x[j] = __fmul2_rn(make_float2(__uint_as_float(v0[2 * j]), __uint_as_float(v0[2 * j + 1])),
                          make_float2(sc, sc));
        x[16 + j] =
            __fmul2_rn(make_float2(__uint_as_float(v1[2 * j]), __uint_as_float(v1[2 * j + 1])),
                       make_float2(sc, sc));
      }
      const int kb = t.b * kKeysT + hf * 64;  // first key of this half
      if (kb + 64 > lim) {  // the causal diagonal or the end of the context
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (kb + 2 * j >= lim) x[j].x = neg_inf();
          if (kb + 2 * j + 1 >= lim) x[j].y = neg_inf();
        }
      }
      float mx;
      {
        float m8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          float mu = fmaxf(x[u].x, x[u].y);
          float mv;
          asm("max.f32 %0, %1, %2, %3;" : "=f"(mv) : "f"(x[8 + u].x), "f"(x[8 + u].y), "f"(mu));
          asm("max.f32 %0, %1, %2, %3;" : "=f"(mu) : "f"(x[16 + u].x), "f"(x[16 + u].y), "f"(mv));
          asm("max.f32 %0, %1, %2, %3;" : "=f"(mv) : "f"(x[24 + u].x), "f"(x[24 + u].y), "f"(mu));
          m8[u] = mv;
        }
        float m3a, m3b;
        asm("max.f32 %0, %1, %2, %3;" : "=f"(m3a) : "f"(m8[0]), "f"(m8[1]), "f"(m8[2]));
        asm("max.f32 %0, %1, %2, %3;" : "=f"(m3b) : "f"(m8[3]), "f"(m8[4]), "f"(m8[5]));
        asm("max.f32 %0, %1, %2, %3;" : "=f"(mx) : "f"(m8[6]), "f"(m8[7]), "f"(m3a));
        mx = fmaxf(mx, m3b);
      }
      float alpha = 1.f;
      bool rescale = false;
      if (m_ref == neg_inf()) {
        m_ref = mx;  // nothing accumulated yet (O and l are zero)
      } else if (mx > m_ref + kRescaleLog2) {
        alpha = ex2(m_ref - mx);
        m_ref = mx;
        rescale = true;
      }
      const float ref = m_ref == neg_inf() ? 0.f : m_ref;
      const float2 nref = make_float2(-ref, -ref);
      float2 acc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
      uint32_t pk[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float2 d = __fadd2_rn(x[j], nref);
        const float2 e = make_float2(ex2(d.x), ex2(d.y));
        acc[j & 3] = __fadd2_rn(acc[j & 3], e);
        pk[j] = cvt_bf16x2(e.x, e.y);
      }
      const float2 s01 = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
      l = fmaf(l, alpha, s01.x + s01.y);
      // the previous PV must be done before P is replaced, O is rescaled or the
      // previous piece's O is read
      if (i > 0 && !wait(B_ODONE, (uint32_t)(i - 1) & 1u)) break;
      tc_fence_after();
      if (pend && !flush()) break;
      if (rescale && !first) {
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t v[32];
          const uint32_t ta = tO + (uint32_t)hf * 128u + (uint32_t)cc * 32u;
          tmem_ld32(ta, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
          tmem_st32(ta, v);
        }
      }
      // P row r, keys of half hf, over the S columns this thread has read
      tmem_st32(tS, pk);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      // keys past the context may hold anything (even NaN): zero their V rows
      // so that P = 0 never meets them (thread (r, hf) clears half hf of key row r)
      const int key0 = t.b * kKeysT;
      if (key0 + kKeysT > c && key0 + r >= c) {
        if (!wait(B_VFULL + sb, (uint32_t)(i >> 1) & 1u)) break;
        unsigned char* vrow = smem + kOffKV + sb * 2 * kOpBytes + kOpBytes + hf * kHalfT + r * 128;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          *reinterpret_cast<uint4*>(vrow + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive(bar(B_PFULL));

      if (last) {
        // hand (m, l) of this half to the partner thread; O is written out
        // during the next tile (or after the loop)
        float* mine = lx + ((np & 1) * 2 + hf) * kRowsT * 2 + r * 2;
        mine[0] = m_ref;
        mine[1] = l;
        mbar_arrive(bar(B_LX + (np & 1)));
        pend = true;
        pend_np = np++;
        pend_m = m_ref;
        pend_l = l;
        pend_complete = (piece_b0 == 0) && (t.b == t.nt - 1);
        pend_orow = valid ? out_row(a, (int64_t)P.qstart[t.s] + tok, t.h * G + r % G) : 0;
        pend_valid = valid && pend_orow >= 0;
        pend_slot = (size_t)w * 2 + (piece_first ? 0 : 1);
      }
      if (idx + 1 < R1) advance(P, S, Hkv, t);
    }
    if (pend && !*abort_flag && wait(B_ODONE, (uint32_t)(i - 1) & 1u)) {
      tc_fence_after();
      flush();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
}

// Merge the pieces of (sequence, query tile, KV head) segments cut between
// CTAs. Grid (CTA boundary, quarter of the tile's rows); eight lanes per
// query row, so each piece's row is one coalesced 512-byte read and a warp has
// four rows' loads in flight. The plan is rebuilt (the prefill grid does not
// change it) before the wait for that grid.
constexpr int kFixRowsPerCta = 32;
constexpr int kFixThreads = 256;

__global__ void __launch_bounds__(kFixThreads)
    prefill_tc_fixup_kernel(const TcArgs a) {
  // the next grid in the stream may start its own preparation now; it waits
  // for this grid before it reads anything this grid writes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ __align__(16) unsigned char fx_smem[];
  PlanSmem P;
  plan_view(fx_smem, a, P);
  PlanInputs in;
  plan_inputs(a, in);
  const int max_workers = prefill_workers(a, fx_smem);
  build_plan(in, P, nullptr);
  const PieceCut cut = build_piece_cut(P, a.Hkv, max(max_workers, 1), kPieceCost4, cut_view(fx_smem, a));
  const int w = blockIdx.x;
  const MergeJob job = merge_job_of(P, a.S, a.Hkv, w, cut.nw, cut);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!job.valid) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int q0 = P.qstart[job.s], lq = P.qstart[job.s + 1] - q0;
  const int npieces = job.last - w + 2;  // workers w-1 .. last
  auto slot_of = [&](int i) -> size_t {
    return (size_t)(w - 1 + i) * 2 + (i == 0 ? job.slot_prev : 0);
  };
  // a warp merges four rows at once: eight lanes per row, sixteen dims per lane
  const int r = blockIdx.y * kFixRowsPerCta + warp * 4 + (lane >> 3);
  const int d0 = (lane & 7) * 16;
  const int tok = job.qt * a.QTb + r / a.G;
  if (tok >= lq) return;
  // online merge over the pieces, four at a time with all their loads in flight
  float m = neg_inf(), sum = 0.f;
  float acc[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j] = 0.f;
  for (int i0 = 0; i0 < npieces; i0 += 4) {
    float li[4];
    float4 x[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      li[u] = neg_inf();
      x[u][0] = x[u][1] = x[u][2] = x[u][3] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i0 + u < npieces) {
        const size_t sl = slot_of(i0 + u);
        li[u] = a.part_lse[sl * kRowsT + r];
        const float4* src =
            reinterpret_cast<const float4*>(a.part_o + (sl * kRowsT + r) * kHeadDim + d0);
#pragma unroll
        for (int k = 0; k < 4; ++k) x[u][k] = src[k];
      }
    }
    const float mn = fmaxf(fmaxf(m, fmaxf(li[0], li[1])), fmaxf(li[2], li[3]));
    if (mn == neg_inf()) continue;
    const float shrink = m == neg_inf() ? 0.f : ex2((m - mn) * kLog2e);
    sum *= shrink;
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] *= shrink;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float wt = li[u] == neg_inf() ? 0.f : ex2((li[u] - mn) * kLog2e);
      sum += wt;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[4 * k + 0] = fmaf(wt, x[u][k].x, acc[4 * k + 0]);
        acc[4 * k + 1] = fmaf(wt, x[u][k].y, acc[4 * k + 1]);
        acc[4 * k + 2] = fmaf(wt, x[u][k].z, acc[4 * k + 2]);
        acc[4 * k + 3] = fmaf(wt, x[u][k].w, acc[4 * k + 3]);
      }
    }
    m = mn;
  }
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j] *= inv;
  const float LSE = sum > 0.f ? m + lg2(sum) * kLn2 : neg_inf();
  const int64_t orow = out_row(a, (int64_t)q0 + tok, job.h * a.G + r % a.G);
  if (orow < 0) return;
  if (a.rows.o) {
    float4* dst = reinterpret_cast<float4*>(a.rows.o + (orow * a.rows.stride + a.rows.slot) * kHeadDim + d0);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      dst[k] = make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
    if ((lane & 7) == 0) a.rows.lse[orow * a.rows.stride + a.rows.slot] = LSE;
    return;
  }
  uint4* dst = reinterpret_cast<uint4*>(a.out + orow * kHeadDim + d0);
  dst[0] = make_uint4(cvt_bf16x2(acc[0], acc[1]), cvt_bf16x2(acc[2], acc[3]),
                      cvt_bf16x2(acc[4], acc[5]), cvt_bf16x2(acc[6], acc[7]));
  dst[1] = make_uint4(cvt_bf16x2(acc[8], acc[9]), cvt_bf16x2(acc[10], acc[11]),
                      cvt_bf16x2(acc[12], acc[13]), cvt_bf16x2(acc[14], acc[15]));
  if ((lane & 7) == 0 && a.lse) a.lse[orow] = LSE;
}

// 3-D view of q as [Tq][Hq][128] bf16, boxes of (128/G) tokens x G heads x 64 dims,
// 128-byte swizzle: one box lands as 128 rows (token-major, head-minor) of 128 B.
bool make_q_map(CUtensorMap* map, const void* q, int64_t num_q_tokens, int Hq, int G, int QTb) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)Hq, (cuuint64_t)num_q_tokens};
  cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)Hq * kHeadDim * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)QTb};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// plan arrays, then the worker starts of the cut, then the split's two words
size_t plan_bytes(int S, int npairs_cap, int workers) {
  return sizeof(int) * ((size_t)npairs_cap + 1 + 3 * ((size_t)S + 1) + (size_t)workers + 1) + 24;
}

}  // namespace

int prefill_tc_geometry(const pa_shape* sh, int64_t num_q_tokens, int max_q_len,
                        PrefillTcGeometry* g, int min_q_len, int max_ctas) {
  DeviceInfo dev;
  if (!current_device_info(&dev)) return PA_ERR_CUDA;
  const int G = sh->num_q_heads / sh->num_kv_heads;
  if (G > kRowsT || kRowsT % G != 0 || max_q_len < min_q_len || max_q_len < 1) {
    g->enabled = false;
    g->ws_bytes = 0;
    return PA_OK;
  }
  const int QTb = kRowsT / G, S = sh->num_seqs;
  const int64_t cap1 = (int64_t)S * ((max_q_len + QTb - 1) / QTb);
  const int64_t cap2 = (num_q_tokens + QTb - 1) / QTb + S;
  const int64_t cap = cap1 < cap2 ? cap1 : cap2;
  if (cap > (1 << 20)) return PA_ERR_UNSUPPORTED;
  g->enabled = true;
  g->npairs_cap = (int)(cap < 1 ? 1 : cap);
  g->QTb = QTb;
  // one CTA per SM (shared memory and TMEM limit it to one)
  g->grid = max_ctas > 0 && max_ctas < dev.num_sms ? max_ctas : dev.num_sms;
  g->workers = g->grid;
  g->smem = 1024 + kOffPlan + round_up(plan_bytes(S, g->npairs_cap, g->workers), 16);
  g->fixup_smem = plan_bytes(S, g->npairs_cap, g->workers);
  if (g->smem > (size_t)dev.max_smem_optin || g->fixup_smem > (size_t)dev.max_smem_optin)
    return PA_ERR_UNSUPPORTED;
  if (!raise_smem_limit(reinterpret_cast<const void*>(paged_prefill_tc_kernel)))
    return PA_ERR_CUDA;
  if (g->fixup_smem > 48 * 1024 &&
      !raise_smem_limit(reinterpret_cast<const void*>(prefill_tc_fixup_kernel)))
    return PA_ERR_CUDA;
  g->ws_lse = round_up(sizeof(float) * 2 * kRowsT * (size_t)g->workers, 256);
  g->ws_o = round_up(sizeof(float) * 2 * kRowsT * kHeadDim * (size_t)g->workers, 256);
  g->ws_bytes = g->ws_lse + g->ws_o;
  return PA_OK;
}

int launch_prefill_tc(const PrefillTcGeometry& g, const pa_bf16* q, const pa_bf16* k_cache,
                      const pa_bf16* v_cache, const int32_t* block_tables,
                      const int32_t* context_lens, const int32_t* cu_seqlens_q,
                      int64_t num_q_tokens, int causal, float scale, pa_bf16* out, float* lse,
                      const pa_shape* sh, void* workspace, cudaStream_t st, int min_q_len,
                      const RowsOut* rows, const int32_t* row_map, int parts, int split) {
  const int G = sh->num_q_heads / sh->num_kv_heads;
  CUtensorMap tmq, tmk, tmv;
  const int64_t pool_rows = sh->num_blocks * sh->num_kv_heads * kBlock;
  if (!make_q_map(&tmq, q, num_q_tokens, sh->num_q_heads, G, g.QTb) ||
      !make_pool_map(&tmk, k_cache, pool_rows) || !make_pool_map(&tmv, v_cache, pool_rows))
    return PA_ERR_CUDA;
  TcArgs a;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.cu_seqlens_q = cu_seqlens_q;
  a.out = out;
  a.lse = lse;
  a.scale_log2 = (float)((double)scale * 1.4426950408889634);
  a.S = sh->num_seqs;
  a.Hq = sh->num_q_heads;
  a.Hkv = sh->num_kv_heads;
  a.G = G;
  a.QTb = g.QTb;
  a.max_blocks = sh->max_blocks_per_seq;
  a.num_blocks = sh->num_blocks;
  a.num_q_tokens = num_q_tokens;
  a.causal = causal ? 1 : 0;
  a.npairs_cap = g.npairs_cap;
  a.num_workers = g.workers;
  a.split = split > 0 ? g.grid : 0;
  a.min_lq = min_q_len;
  if (rows) a.rows = *rows;
  a.row_map = row_map;
  char* ws = static_cast<char*>(workspace);
  a.part_lse = reinterpret_cast<float*>(ws);
  a.part_o = reinterpret_cast<float*>(ws + g.ws_lse);
  if ((parts & 1) && launch_dependent(paged_prefill_tc_kernel, dim3(g.grid), dim3(kThreadsT),
                                      g.smem, st, tmq, tmk, tmv, a) != cudaSuccess)
    return PA_ERR_CUDA;
  if ((parts & 2) && launch_dependent(prefill_tc_fixup_kernel, dim3(g.workers, kRowsT / kFixRowsPerCta),
                       dim3(kFixThreads), g.fixup_smem, st, a) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

unsigned take_error_word_prefill(cudaStream_t stream, int* rc) {
  unsigned v = 0, zero = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess ||
      cudaMemcpyFromSymbol(&v, g_pa_error_word, sizeof v) != cudaSuccess ||
      cudaMemcpyToSymbol(g_pa_error_word, &zero, sizeof zero) != cudaSuccess) {
    *rc = PA_ERR_CUDA;
    return 0;
  }
  return v;
}

}  // namespace pa
