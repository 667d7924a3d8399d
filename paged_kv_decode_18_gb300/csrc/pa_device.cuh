// pa_device.cuh -- device-side building blocks shared by the kernels of
// libpagedattn (sm_103a): asynchronous-copy and mbarrier wrappers, the
// tensor-core fragments, the device error word, and the per-CTA work plan
// that cuts a batch of paged sequences into equal tile ranges.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

constexpr int kHeadDim = 128;                        // built head_dim
constexpr int kBlock = 16;                           // built block_size (tokens)
constexpr int kTileBytes = kBlock * kHeadDim * 2;    // one (block, kv head) K or V tile
// one (block, kv head) tile of the int8 pool: 16 x 128 codes, then the 16 rows'
// fp32 scales (a multiple of 16 bytes, so every tile is a bulk-copy source)
constexpr int kInt8TileBytes = kBlock * kHeadDim + kBlock * 4;
static_assert(kInt8TileBytes == PA_INT8_TILE_BYTES, "int8 tile layout");
static_assert(kInt8TileBytes % 16 == 0, "int8 tiles must stay 16-byte aligned");
constexpr unsigned kFull = 0xffffffffu;

// Time limit of every wait on an asynchronous copy. A copy that has not landed
// by then sets PA_DEVERR_PIPE_TIMEOUT and the waiting warp gives up.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

// ---------------------------------------------------------------------------
// device error word: one per translation unit (each TU owns its copy and
// exposes a host reader), OR-ed together by pa_debug_read_error.
// ---------------------------------------------------------------------------
static __device__ unsigned int g_pa_error_word = 0;

__device__ __forceinline__ void flag_error(unsigned bits) {
  atomicOr(&g_pa_error_word, bits);
}

// ---------------------------------------------------------------------------
// small PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of an mbarrier. Returns false (and flags
// PA_DEVERR_PIPE_TIMEOUT) if the phase did not complete within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      flag_error(PA_DEVERR_PIPE_TIMEOUT);
      return false;
    }
  }
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy / TMA) writes to the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier.
// dst/src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 2-D tiled TMA load (tensor map in kernel parameter space) into shared
// memory, completion counted on an mbarrier. x (innermost) in elements.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// fast exp2 / log2 (PTX approximate instructions; relative error ~2^-22)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// bf16 pair (one 32-bit word) -> two floats: low element, high element.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// float -> bf16 bits, round to nearest even (NaN kept NaN).
__device__ __forceinline__ uint32_t f2bf_bits(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0u;
  u += 0x7fffu + ((u >> 16) & 1u);
  return u >> 16;
}

__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  return f2bf_bits(lo) | (f2bf_bits(hi) << 16);
}

// ---------------------------------------------------------------------------
// tensor-core fragments (mma.sync m16n8k16, bf16 x bf16 -> fp32)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// A pure register operation: not volatile, so the compiler may interleave
// independent products with other work.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// Work plan.
//
// The batch is a list of (sequence, query tile) pairs; pair p needs n_p K/V
// tiles (16 keys each) for each of the Hkv KV heads. Flat tile index order is
// (pair, kv head, tile), so every (pair, kv head) -- a "segment" -- is a
// contiguous run of n_p indices. pair_off[p] = Hkv * sum_{p' < p} n_p'. Each
// CTA rebuilds this prefix in its shared memory from context_lens and
// cu_seqlens_q (a few KB), so no separate planning kernel or host sync is
// needed; warps then locate their ranges by binary search.
// ---------------------------------------------------------------------------
struct PlanSmem {
  int* pair_off;   // [npairs_cap + 1]
  int* seq_pair;   // [S + 1]  first pair of each sequence
  int* ctx;        // [S]      context length (validated)
  int* qstart;     // [S + 1]  cu_seqlens_q (validated)
  int npairs;
  int total;       // total flat tiles
};

struct PlanInputs {
  const int32_t* context_lens;  // [S]
  const int32_t* cu_seqlens_q;  // [S + 1] or nullptr (decode: one query per sequence)
  int S;
  int Hkv;
  int max_ctx;       // max_blocks_per_seq * block size
  int qtile;         // query tokens per tile (1 for decode)
  int causal;
  int npairs_cap;
  int64_t num_q_rows;  // rows of q / out; every sequence's rows must lie inside
  int key_tile = kBlock;       // keys per flat tile (a multiple of the block size)
  int min_lq = 0;              // sequences whose q_len lies outside [min_lq, max_lq]
  int max_lq = 0x7fffffff;     // belong to another kernel: no tiles here (not an error)
  // decode only: every sequence is cut into `parts` near-equal block ranges,
  // one pair each (pair s * parts + j holds blocks part_begin(j) ..), the
  // split-K partitions; 1 = one pair per sequence
  int parts = 1;
};

// First block of partition j of a sequence with nt blocks cut into `parts`.
__device__ __forceinline__ int part_begin(int j, int nt, int parts) {
  return (int)(((long long)j * nt) / parts);
}

// Exclusive scan of n ints in shared memory, in place, by warp 0 of the CTA
// (each lane scans a contiguous chunk, then the lanes' totals are scanned by
// shuffles). The caller synchronises the CTA before and after. Returns the
// total in warp 0's lanes.
__device__ inline int warp0_exclusive_scan(int* data, int n) {
  const int lane = threadIdx.x & 31;
  const int chunk = (n + 31) / 32;
  const int b = min(n, lane * chunk), e = min(n, b + chunk);
  int local = 0;
  for (int i = b; i < e; ++i) local += data[i];
  int x = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  const int total = __shfl_sync(kFull, x, 31);
  int run = x - local;
  for (int i = b; i < e; ++i) {
    const int v = data[i];
    data[i] = run;
    run += v;
  }
  return total;
}

// Number of key tiles query tile qt of sequence s needs (per KV head).
__device__ __forceinline__ int pair_tiles(int c, int lq, int qt, int qtile, int causal,
                                          int key_tile = kBlock) {
  int kv_end = causal ? (c - lq + min(qtile * (qt + 1), lq)) : c;
  return (kv_end + key_tile - 1) / key_tile;
}

// Build the plan in shared memory. All threads of the CTA must call it; it
// ends with a CTA barrier. Invalid lengths are clamped (and flagged) so that
// every later access stays inside the caller's buffers.
//
// Decode (no cu_seqlens_q): pair p is sequence p (a sequence with an empty
// context is a pair with no tiles), so one scan suffices.
__device__ inline void build_plan(const PlanInputs& in, PlanSmem& P, int* /*scratch*/) {
  const int tid = threadIdx.x, nthreads = blockDim.x;
  const int S = in.S;
  const bool varlen = in.cu_seqlens_q != nullptr;
  for (int s = tid; s < S; s += nthreads) {
    int c = in.context_lens[s];
    if (c < 0 || c > in.max_ctx) {
      flag_error(PA_DEVERR_CONTEXT_RANGE);
      c = c < 0 ? 0 : in.max_ctx;
    }
    P.ctx[s] = c;
    if (varlen) {
      const int q0 = in.cu_seqlens_q[s];
      int lq = in.cu_seqlens_q[s + 1] - q0;
      // causal: a query window cannot be longer than its context; non-causal
      // queries see the whole (non-empty) context whatever their number
      if (lq < 0 || (lq > c && (in.causal || c == 0)) || q0 < 0 ||
          (int64_t)q0 + lq > in.num_q_rows) {
        flag_error(PA_DEVERR_QLEN_RANGE);
        lq = 0;  // the sequence produces no rows
      }
      if (lq < in.min_lq || lq > in.max_lq) lq = 0;  // handled by another kernel
      P.qstart[s] = q0;
      P.seq_pair[s] = (lq + in.qtile - 1) / in.qtile;  // query tiles of s
      if (s == S - 1) P.qstart[S] = in.cu_seqlens_q[S];
    } else if (in.parts <= 1) {
      P.qstart[s] = s;
      P.seq_pair[s] = s;
      P.pair_off[s] = in.Hkv * ((c + kBlock - 1) / kBlock);
      if (s == S - 1) {
        P.qstart[S] = S;
        P.seq_pair[S] = S;
      }
    } else {
      const int nt = (c + kBlock - 1) / kBlock;
      P.qstart[s] = s;
      P.seq_pair[s] = s * in.parts;
      for (int j = 0; j < in.parts; ++j)
        P.pair_off[s * in.parts + j] =
            in.Hkv * (part_begin(j + 1, nt, in.parts) - part_begin(j, nt, in.parts));
      if (s == S - 1) {
        P.qstart[S] = S;
        P.seq_pair[S] = S * in.parts;
      }
    }
  }
  __syncthreads();
  int npairs = varlen || in.parts <= 1 ? S : S * in.parts;
  if (varlen) {
    if (tid < 32) {
      const int n = warp0_exclusive_scan(P.seq_pair, S);
      if (tid == 0) P.seq_pair[S] = n;
    }
    __syncthreads();
    npairs = P.seq_pair[S];
    if (npairs > in.npairs_cap) {
      if (tid == 0) flag_error(PA_DEVERR_PLAN_OVERFLOW);
      npairs = 0;  // do nothing rather than overflow the shared arrays
    }
    for (int s = tid; s < S; s += nthreads) {
      const int p0 = P.seq_pair[s], p1 = P.seq_pair[s + 1];
      if (p1 > npairs) continue;
      const int c = P.ctx[s];
      const int q0 = in.cu_seqlens_q[s];
      int lq = in.cu_seqlens_q[s + 1] - q0;
      if (lq < 0 || (lq > c && (in.causal || c == 0)) || q0 < 0 ||
          (int64_t)q0 + lq > in.num_q_rows)
        lq = 0;
      if (lq < in.min_lq || lq > in.max_lq) lq = 0;
      for (int p = p0; p < p1; ++p)
        P.pair_off[p] = in.Hkv * pair_tiles(c, lq, p - p0, in.qtile, in.causal, in.key_tile);
    }
    __syncthreads();
  }
  if (tid < 32) {
    const int total = warp0_exclusive_scan(P.pair_off, npairs);
    if (tid == 0) P.pair_off[npairs] = total;
  }
  __syncthreads();
  P.npairs = npairs;
  P.total = P.pair_off[npairs];
}

// Largest i in [lo, hi) with a[i] <= x (a non-decreasing, a[lo] <= x).
__device__ __forceinline__ int upper_index(const int* a, int lo, int hi, int x) {
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (a[mid] <= x)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

// Position of one flat tile index.
struct TilePos {
  int s;    // sequence
  int p;    // pair (sequence, query tile)
  int qt;   // query tile within the sequence
  int h;    // kv head
  int b;    // key tile (block) within the segment
  int nt;   // key tiles of the segment
};

__device__ __forceinline__ TilePos locate(const PlanSmem& P, int S, int Hkv, int idx) {
  TilePos t;
  t.p = upper_index(P.pair_off, 0, P.npairs, idx);
  t.s = upper_index(P.seq_pair, 0, S, t.p);
  t.qt = t.p - P.seq_pair[t.s];
  t.nt = (P.pair_off[t.p + 1] - P.pair_off[t.p]) / Hkv;
  const int local = idx - P.pair_off[t.p];
  t.h = local / t.nt;
  t.b = local - t.h * t.nt;
  return t;
}

// Position of flat tile idx >= from's index, found by scanning forward from
// `from` (a nearby position, usually the same or the next few pairs), which
// is much cheaper than a binary search when idx is close.
__device__ __forceinline__ TilePos locate_from(const PlanSmem& P, int Hkv, const TilePos& from,
                                               int idx) {
  TilePos t = from;
  while (P.pair_off[t.p + 1] <= idx) ++t.p;
  while (P.seq_pair[t.s + 1] <= t.p) ++t.s;
  t.qt = t.p - P.seq_pair[t.s];
  t.nt = (P.pair_off[t.p + 1] - P.pair_off[t.p]) / Hkv;
  const int local = idx - P.pair_off[t.p];
  t.h = local / t.nt;
  t.b = local - t.h * t.nt;
  return t;
}

// Start of worker w's range when W flat tiles are cut into nw equal
// contiguous ranges: floor(w * W / nw).
__device__ __forceinline__ int range_start(int w, int W, int nw) {
  return (int)(((long long)w * W) / nw);
}

// The equal cut as an object: worker w starts at range_start(w); tile x is held
// by worker floor(((x + 1) * nw - 1) / W).
struct EqualCut {
  int W, nw;
  __device__ __forceinline__ int start(int w) const { return range_start(w, W, nw); }
  __device__ __forceinline__ int owner(int x) const {
    return (int)(((long long)(x + 1) * nw - 1) / W);
  }
};

// A cut that charges every segment start `cost4`/4 of a tile on top of the
// tiles themselves (starting a segment costs its query tile, a first score
// tile with nothing to overlap, and a write-out), so a worker whose range
// holds many short segments gets fewer tiles. The cost of tiles 0 .. x-1 is
// 4x + cost4 * (segment starts below x); worker w starts at the first x whose
// cost reaches floor(w * C / nw), C the total. The starts live in a shared
// array of nw + 1 entries, built by build_piece_cut.
struct PieceCut {
  const int* cut;  // [nw + 1] first tile of each worker; cut[nw] = total
  int nw;
  __device__ __forceinline__ int start(int w) const { return cut[w]; }
  // largest w with cut[w] <= x: the worker holding tile x
  __device__ __forceinline__ int owner(int x) const { return upper_index(cut, 0, nw, x); }
};

// Build the PieceCut of a plan into cut[0 .. nw] (nw + 1 <= max_workers + 1
// ints). All threads of the CTA call it; it ends with a CTA barrier. Needs
// every pair to hold at least one tile per KV head (true of every query-tile
// plan), so pair p begins after p * Hkv segment starts: its tiles cost
// base(p) = 4 pair_off[p] + cost4 p Hkv before it. One thread per worker finds
// the pair its target falls in by bisection, then the tile in closed form.
// With nw <= C / (4 + cost4), consecutive targets are at least one tile's
// largest cost apart, so the starts strictly increase: no worker is empty.
__device__ inline PieceCut build_piece_cut(const PlanSmem& P, int Hkv, int max_workers, int cost4,
                                           int* cut) {
  const int tid = threadIdx.x, nthreads = blockDim.x;
  const long long C = 4LL * P.total + (long long)cost4 * P.npairs * Hkv;
  long long nwl = C / (4 + cost4);
  if (nwl > max_workers) nwl = max_workers;
  if (nwl < 1) nwl = 1;
  const int nw = (int)nwl;
  const bool narrow = C * nw < (1LL << 32);  // targets in 32-bit arithmetic
  auto base = [&](int p) -> long long {
    return 4LL * P.pair_off[p] + (long long)cost4 * p * Hkv;
  };
  for (int w = 1 + tid; w < nw; w += nthreads) {
    const long long T = narrow ? (long long)((uint32_t)w * (uint32_t)C / (uint32_t)nw)
                               : ((long long)w * C) / nw;  // 0 < T < C
    // the pair p with base(p) < T <= base(p + 1)
    int lo = 0, hi = P.npairs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (base(mid) < T)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int o0 = P.pair_off[lo];
    const int nt = (P.pair_off[lo + 1] - o0) / Hkv;
    const int D = (int)(T - base(lo));  // 1 .. Hkv (4 nt + cost4)
    const int seg = 4 * nt + cost4;     // cost of one whole segment of this pair
    const int h = (D - 1) / seg;        // the segment it falls in
    const int rem = D - h * seg;        // 1 .. seg
    // tile r (1-based) of segment h costs cost4 + 4r up to and including it
    const int r = max(1, (rem - cost4 + 3) / 4);
    cut[w] = o0 + h * nt + r;
  }
  if (tid == 0) {
    cut[0] = 0;
    cut[nw] = P.total;
  }
  __syncthreads();
  PieceCut c;
  c.cut = cut;
  c.nw = nw;
  return c;
}

// The SMs of one pa_decode_varlen call split between its tensor-core prefill
// grid and its verify grid when the two run side by side: the prefill grid
// keeps K of its N CTAs (one per SM) and the verify grid works on the rest,
// with K = ceil(N A / (A + N V)), which evens out the two halves' times under
// a plain cost model: A = the prefill work in CTA-time (kSplitTileNs per 128
// keys seen by a 128-row query tile), V = the verify grid's time on all N SMs
// (512 bytes of K and V per key seen per KV head at kSplitBytesPerUs). Every
// grid that needs K computes it from the same inputs with the same integer
// arithmetic, so they agree. Sequences with q_len >= min_lq are prefill. All
// threads of the CTA call it (two CTA barriers); red: two 8-byte-aligned
// words of shared memory. Returns 0 (no prefill work) .. N (no verify work).
// A prefill tile beside the HBM-bound verify grid takes longer than alone
// (1.46 us: its K/V loads from L2 wait behind the verify stream); a sweep of
// this constant on the mixed batch (48 verify windows + two 512-token chunks)
// put the best split at 2.25-3.0 us per tile (176-179 us per call against
// 193 us with the grids in turn) and a cliff below it (2.0 us: 188 us), so the
// constant sits on the safe side.
constexpr long long kSplitTileNs = 2500;
constexpr long long kSplitBytesPerUs = 5900000;  // verify grid on all SMs (HBM)

__device__ inline int overlap_split(const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                    int S, int Hkv, int G, int causal, int min_lq, int max_ctx,
                                    int N, unsigned long long* red) {
  if (threadIdx.x == 0) red[0] = red[1] = 0ull;
  __syncthreads();
  unsigned long long pf = 0, vf = 0;  // keys seen, summed over query tiles (one KV head)
  const int qt_pf = 128 / G, qt_v = 16 / G;  // query tokens per tile of either grid
  for (int s = threadIdx.x; s < S; s += blockDim.x) {
    const int c = min(max(context_lens[s], 0), max_ctx);
    const int lq = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
    if (lq <= 0 || c <= 0 || (causal && lq > c)) continue;
    const int qt = lq >= min_lq ? qt_pf : qt_v;
    const long long nq = (lq + qt - 1) / qt;
    // causal: query tile j sees c - lq + min(qt (j + 1), lq) keys
    const long long keys =
        causal ? nq * (c - lq) + (long long)qt * nq * (nq - 1) / 2 + lq : nq * (long long)c;
    if (lq >= min_lq)
      pf += (unsigned long long)keys;
    else
      vf += (unsigned long long)keys;
  }
  if (pf) atomicAdd(&red[0], pf);
  if (vf) atomicAdd(&red[1], vf);
  __syncthreads();
  const long long A = (long long)red[0] * Hkv * kSplitTileNs / 128;
  const long long V = (long long)red[1] * Hkv * 512 * 1000 / kSplitBytesPerUs;
  if (A == 0) return 0;
  if (V == 0) return N;
  const long long K = ((long long)N * A + A + (long long)N * V - 1) / (A + (long long)N * V);
  return (int)(K < 1 ? 1 : (K > N - 1 ? N - 1 : K));
}

// The merge a worker boundary owns. A segment (pair, kv head) cut by range
// boundaries is merged by the first boundary inside it: boundary w owns the
// segment containing tile range_start(w) when that segment began inside worker
// w-1's range. Its pieces are held by workers w-1 .. last: worker w-1 in slot
// slot_prev (0 if the segment starts exactly at w-1's range start, else 1),
// every later worker in slot 0.
struct MergeJob {
  bool valid;
  int s, qt, h, last, slot_prev;
};

template <class Cut>
__device__ inline MergeJob merge_job_of(const PlanSmem& P, int S, int Hkv, int w, int nw,
                                        const Cut& cut) {
  MergeJob j;
  j.valid = false;
  if (w <= 0 || w >= nw) return j;
  const int R0 = cut.start(w);
  if (R0 >= P.total) return j;
  const TilePos t = locate(P, S, Hkv, R0);
  const int A = R0 - t.b;  // flat start of the segment
  const int R0prev = cut.start(w - 1);
  if (t.b == 0 || A < R0prev) return j;
  j.valid = true;
  j.s = t.s;
  j.qt = t.qt;
  j.h = t.h;
  j.last = cut.owner(A + t.nt - 1);  // worker holding the last tile
  j.slot_prev = (A == R0prev) ? 0 : 1;
  return j;
}

__device__ inline MergeJob merge_job(const PlanSmem& P, int S, int Hkv, int w, int W, int nw) {
  return merge_job_of(P, S, Hkv, w, nw, EqualCut{W, nw});
}

// Step a position to the next flat tile (only called while idx + 1 < total).
__device__ __forceinline__ void advance(const PlanSmem& P, int S, int Hkv, TilePos& t) {
  if (++t.b < t.nt) return;
  t.b = 0;
  if (++t.h < Hkv) return;
  t.h = 0;
  do {
    ++t.p;
  } while (P.pair_off[t.p + 1] == P.pair_off[t.p]);
  while (P.seq_pair[t.s + 1] <= t.p) ++t.s;
  t.qt = t.p - P.seq_pair[t.s];
  t.nt = (P.pair_off[t.p + 1] - P.pair_off[t.p]) / Hkv;
}

}  // namespace pa
