// pa_decode.cu -- paged decode attention (one query token per sequence) on
// the CUDA cores, the split-K partial merge, and their C-ABI entry points.
//
// What is computed (LLM inference engine work-log, "KV Cache > The Idea";
// course README "Build an LLM Inference Engine From Scratch", curriculum row
// "Memory & KV Cache" and the claim "online softmax is exact; paged and
// split-K variants agree"): for every sequence s and query head h,
//   out[s,h] = sum_p softmax_p(scale * q[s,h] . K_s[p]) V_s[p],
//   lse[s,h] = ln sum_p exp(scale * q[s,h] . K_s[p]),
// with K_s/V_s reached through the block table and KV head h / 2.
//
// Design (GB300): decode at q_len 1 is an HBM stream -- each K/V element read
// feeds 2 query heads, about 2 flop/byte -- so it runs on the CUDA cores and
// everything is arranged around moving bytes:
//   * one warp is one worker; it owns a contiguous range of (sequence,
//     KV head, block) tiles and a private ring of NSTAGE shared-memory stages;
//   * lane 0 moves each 4 KB K tile and 4 KB V tile of one (block, KV head)
//     with a 1-D bulk async copy (TMA engine) onto the stage's mbarrier, plus
//     the 512 B of the two query heads when a new sequence starts;
//   * both query heads of the KV head share every tile read from shared memory;
//   * QK^T: lane (g, c) holds dims 16c..16c+15 of 4 tokens for both heads;
//     the 8 partial dots are reduce-scattered over 8 lanes (7 shuffles) so
//     each lane ends with one (token, head) score; fp32 pairs run through the
//     packed f32x2 FMA pipe of sm_100+;
//   * online softmax in the log2 domain (scale * log2 e folded into q);
//   * PV: the same lane layout accumulates 2 heads x 16 dims in fp32 pairs;
//     the 4 token groups are combined by a shuffle reduce-scatter once per
//     piece, after the stage has been refilled.
// A batch is cut into equal tile ranges over all resident warps (num_splits
// 0), so ragged batches and long contexts balance; a (sequence, KV head) cut
// by a range boundary leaves partials that a small merge kernel combines.
// The same kernel, templated on the pool format, serves the 8-bit pools
// (int8 or FP8 E4M3 codes, one fp32 scale per (token, KV head) row). There
// the per-value conversions plus fp32 products made the loop issue-bound, so
// both contractions of a tile run on warp MMAs instead (m16n8k16, f16
// operands, fp32 accumulation): the codes become f16 exactly (the hardware
// E4M3 conversion; for int8 a byte permute into the mantissa of the half 1024
// and one packed subtraction), q is scaled by a power of two so it is exact
// in f16, the K row scales multiply the scores, and the V row scales fold
// into the softmax weights (normalised per tile so they fit f16). The integer
// MMA (s8) was measured 1.8x slower on this part: its int8 tensor rate is low.
#include "pa_device.cuh"
#include "pa_host.h"

namespace pa {
namespace {

constexpr int kG = 2;                          // query heads per KV head (built)
constexpr int kQBytes = kG * kHeadDim * 2;     // 512

// Pool element formats of the decode kernel.
enum : int { kFmtBf16 = 0, kFmtI8 = 1, kFmtF8 = 2 };

// Stage layout for a KV element format: the K tile, the V tile, then q (at a
// piece's first tile). A tile is one bulk copy of the pool's (block, KV head)
// run: bf16 [16][128] (4 KB), or 8-bit codes (int8 or FP8 E4M3) [16][128]
// (2 KB) followed by the 16 rows' fp32 scales.
template <int FMT>
struct KvFormat {
  static constexpr bool Q8 = FMT != kFmtBf16;  // one-byte codes with row scales
  static constexpr int kTile = Q8 ? kInt8TileBytes : kTileBytes;  // one K or V tile, bytes
  static constexpr int kScaleOff = kBlock * kHeadDim;            // 8-bit: scales within a tile
  static constexpr int kQOff = 2 * kTile;
  static constexpr int kStage = kQOff + kQBytes;
  static_assert(kTile % 16 == 0 && kStage % 16 == 0, "bulk copies need 16-byte alignment");
  static_assert(!Q8 || kScaleOff + kBlock * 4 == kTile, "8-bit row scales end the tile");
};

template <int NSTAGE, int FMT>
struct WarpLayout {
  static constexpr int kStageBytes = KvFormat<FMT>::kStage;
  static constexpr int kBarOff = NSTAGE * kStageBytes;
  static constexpr int kPOff = kBarOff + ((NSTAGE * 8 + 15) / 16) * 16;
  static constexpr int kBytes = ((kPOff + 128 + 127) / 128) * 128;
};

enum : int { kBalanced = 0, kFixed = 1 };

struct DecodeArgs {
  const uint16_t* q;
  const unsigned char* k_cache;  // bf16, int8 or FP8 tiles (KvFormat)
  const unsigned char* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  uint16_t* out;
  float* lse;
  float scale_log2;
  int S, Hq, Hkv, max_blocks;
  int64_t num_blocks;
  int mode;         // kBalanced or kFixed
  int num_splits;   // kFixed: P
  int num_workers;  // kBalanced: warps launched
  int parts;        // kBalanced: split-K partitions per sequence (1: none); with
                    // parts > 1 finished partitions go to `rows` in slot = partition
  float* part_o;    // kBalanced: [NW*2][G][D]; kFixed: [S][Hq][P][D]
  float* part_lse;  // kBalanced: [NW*2][G];    kFixed: [S][Hq][P]
  int early;        // 1: plan and table reads may run before the previous grid ends
  // fp32 row output (balanced mode only): when rows_o is set, finished rows go
  // to rows_o[(row * rows_stride + rows_slot) * D] and rows_lse[row *
  // rows_stride + rows_slot] (normalised o and lse, as one split-K partial)
  // instead of out / lse
  RowsOut rows;
  int skip_copy;    // failure-detection hook: flat tile whose copy is left out (-1: none)
  // 1: the previous grid is not waited for before the work (the grid ahead of
  // it has already been waited for by every CTA of that previous grid); thread
  // 0 of each CTA waits for it only on the way out, so that this grid never
  // completes before it (the cascade's suffix half, beside its prefix half)
  int late;
};

// Write 8 dims (one lane's chunk) of one output row as bf16.
__device__ __forceinline__ void store_out8(uint16_t* dst, const float (&v)[8], float inv) {
  uint4 o;
  o.x = pack_bf2(v[0] * inv, v[1] * inv);
  o.y = pack_bf2(v[2] * inv, v[3] * inv);
  o.z = pack_bf2(v[4] * inv, v[5] * inv);
  o.w = pack_bf2(v[6] * inv, v[7] * inv);
  *reinterpret_cast<uint4*>(dst) = o;
}

__device__ __forceinline__ void store_f8(float* dst, const float (&v)[8], float inv) {
  reinterpret_cast<float4*>(dst)[0] = make_float4(v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv);
  reinterpret_cast<float4*>(dst)[1] = make_float4(v[4] * inv, v[5] * inv, v[6] * inv, v[7] * inv);
}

// Merge the pieces of one cut (sequence, KV head) segment -- the a7 formula
// over workers w-1 .. job.last -- and write its two output rows. One warp.
// Partials are read through L2 (ld.global.cg): other SMs wrote them. The
// log-sum-exps and vectors of up to eight pieces are loaded together, so a
// typical cut costs one round trip to L2.
constexpr int kMergeChunk = 8;

__device__ __forceinline__ void merge_segment(const MergeJob& job, int w, int lane,
                                              const float* __restrict__ part_o,
                                              const float* __restrict__ part_lse, int Hq,
                                              uint16_t* __restrict__ out,
                                              float* __restrict__ lse, const RowsOut& rows) {
  const int s = job.s, h = job.h, last = job.last, slot_prev = job.slot_prev;
  const int npieces = last - w + 2;  // workers w-1 .. last
  auto slot_of = [&](int i) -> size_t {
    return (size_t)(w - 1 + i) * 2 + (i == 0 ? slot_prev : 0);
  };
  float4 acc[kG];
  for (int g = 0; g < kG; ++g) acc[g] = make_float4(0.f, 0.f, 0.f, 0.f);
  // each round handles kMergeChunk pieces: lane i holds piece i's lse values
  float mx[kG] = {neg_inf(), neg_inf()}, sum[kG] = {0.f, 0.f};
  for (int i0 = 0; i0 < npieces; i0 += kMergeChunk) {
    const int n = min(kMergeChunk, npieces - i0);
    float li[kG] = {neg_inf(), neg_inf()};
    if (lane < n) {
      const float2 v = __ldcg(reinterpret_cast<const float2*>(part_lse + slot_of(i0 + lane) * kG));
      li[0] = v.x;
      li[1] = v.y;
    }
    float4 o[kMergeChunk][kG];
#pragma unroll
    for (int j = 0; j < kMergeChunk; ++j) {
#pragma unroll
      for (int g = 0; g < kG; ++g) {
        o[j][g] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < n)
          o[j][g] = __ldcg(reinterpret_cast<const float4*>(
              part_o + (slot_of(i0 + j) * kG + g) * kHeadDim + lane * 4));
      }
    }
    float e[kG];
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      float m = li[g];
#pragma unroll
      for (int x = 16; x > 0; x >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, x));
      m = fmaxf(m, mx[g]);
      // rescale what earlier rounds accumulated to the new maximum
      const float r = ex2((mx[g] - m) * kLog2e);
      sum[g] *= r;
      acc[g].x *= r; acc[g].y *= r; acc[g].z *= r; acc[g].w *= r;
      e[g] = ex2((li[g] - m) * kLog2e);  // unnormalised weight of piece lane
      float t = e[g];
#pragma unroll
      for (int x = 16; x > 0; x >>= 1) t += __shfl_xor_sync(kFull, t, x);
      sum[g] += t;
      mx[g] = m;
    }
#pragma unroll
    for (int j = 0; j < kMergeChunk; ++j) {
#pragma unroll
      for (int g = 0; g < kG; ++g) {
        const float wt = __shfl_sync(kFull, e[g], j);
        acc[g].x = fmaf(wt, o[j][g].x, acc[g].x);
        acc[g].y = fmaf(wt, o[j][g].y, acc[g].y);
        acc[g].z = fmaf(wt, o[j][g].z, acc[g].z);
        acc[g].w = fmaf(wt, o[j][g].w, acc[g].w);
      }
    }
  }
  float LSE[kG];
#pragma unroll
  for (int g = 0; g < kG; ++g) {
    LSE[g] = mx[g] + lg2(sum[g]) * kLn2;
    const float inv = 1.f / sum[g];
    acc[g].x *= inv; acc[g].y *= inv; acc[g].z *= inv; acc[g].w *= inv;
  }
#pragma unroll
  for (int g = 0; g < kG; ++g) {
    const size_t row = (size_t)s * Hq + (size_t)h * kG + g;
    if (rows.o) {
      const size_t r = row * rows.stride + rows.slot;
      *reinterpret_cast<float4*>(rows.o + r * kHeadDim + lane * 4) = acc[g];
      if (lane == 0) rows.lse[r] = LSE[g];
      continue;
    }
    uint2 o;
    o.x = pack_bf2(acc[g].x, acc[g].y);
    o.y = pack_bf2(acc[g].z, acc[g].w);
    *reinterpret_cast<uint2*>(out + row * kHeadDim + lane * 4) = o;
    if (lse && lane == 0) lse[row] = LSE[g];
  }
}

// The 16 dims 16*c8 .. 16*c8+15 of one bf16 token row in stage memory, as 8 pairs.
__device__ __forceinline__ void load_row16(const unsigned char* row, float2 (&f)[8]) {
  const uint4 wa = *reinterpret_cast<const uint4*>(row);
  const uint4 wb = *reinterpret_cast<const uint4*>(row + 16);
  const uint32_t wk[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
  for (int j = 0; j < 8; ++j) f[j] = make_float2(bf_lo(wk[j]), bf_hi(wk[j]));
}

// Two floats -> an f16 pair (lo in the low half), rounded to nearest even.
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Four 8-bit codes (bytes 0..3 of w) -> two f16 pairs, exactly: (byte 0, 1)
// in lo, (byte 2, 3) in hi. FP8 E4M3: the hardware conversion (every E4M3
// value is a normal half; the NaN codes become NaN). int8: the byte, biased
// by 128, becomes the low mantissa bits of the half 1024; one packed
// subtraction of 1152 leaves the code.
template <int FMT>
__device__ __forceinline__ void codes_to_h2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  if constexpr (FMT == kFmtF8) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
  } else {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t blo = __byte_perm(u, 0x64646464u, 0x4140u);
    const uint32_t bhi = __byte_perm(u, 0x64646464u, 0x4342u);
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(blo), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(bhi), "r"(0x64806480u));
  }
}

// d += A * B for one m16n8k16 tile: A row-major 16 x 16 f16 (a0: row g, k
// 2c..2c+1; a1: row g+8, same k; a2: row g, k 2c+8..2c+9; a3: row g+8), B
// 16 x 8 f16 (b0: k 2c..2c+1, column g; b1: k 2c+8..2c+9), fp32 d (d0, d1:
// row g, columns 2c, 2c+1; d2, d3: row g+8), where g = lane / 4, c = lane % 4.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int NWARPS, int NSTAGE, int FMT>
__global__ void __launch_bounds__(NWARPS * 32, FMT != kFmtBf16 || NWARPS <= 6 ? 2 : 1)
    paged_decode_kernel(const DecodeArgs a) {
  using L = WarpLayout<NSTAGE, FMT>;
  using F = KvFormat<FMT>;
  constexpr bool Q8 = F::Q8;
  constexpr int kStageBytes = F::kStage;
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned char* wbuf = smem + warp * L::kBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(wbuf + L::kBarOff);
  const int S = a.S, Hkv = a.Hkv, Hq = a.Hq;

  int* pm = reinterpret_cast<int*>(smem + NWARPS * L::kBytes);
  const int parts = a.mode == kBalanced ? a.parts : 1;
  PlanSmem P;
  P.pair_off = pm;
  P.seq_pair = P.pair_off + (S * parts + 1);
  P.ctx = P.seq_pair + (S + 1);
  P.qstart = P.ctx + S;
  int* scratch = P.qstart + (S + 1);

  if (lane == 0) {
    for (int i = 0; i < NSTAGE; ++i) mbar_init(smem_addr(&bars[i]), 1);
    mbar_fence_init();
  }
  // This grid is launched as a programmatic dependent of the previous one on
  // the stream. By default it waits for that grid right here, before reading
  // anything. With `early` (used only behind this library's own cache-write
  // kernel, which writes nothing but the step's new rows, each in the last
  // block of its sequence's context) the plan and the block-table window are
  // prepared at once and every tile but a segment's last streams in while the
  // write runs: a warp waits for the write only before it copies the last
  // tile of a (sequence, KV head). Thread 0 of CTA 0 also waits once, so
  // that this grid never completes before the write.
  if (!a.early && !a.late) asm volatile("griddepcontrol.wait;" ::: "memory");
  auto late_exit = [&]() {
    if (a.late && threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
  };
  PlanInputs in;
  in.context_lens = a.context_lens;
  in.cu_seqlens_q = nullptr;
  in.S = S;
  in.Hkv = Hkv;
  in.max_ctx = a.max_blocks * kBlock;
  in.qtile = 1;
  in.causal = 1;
  in.npairs_cap = S * parts;
  in.num_q_rows = S;
  in.parts = parts;
  build_plan(in, P, scratch);  // ends with __syncthreads: barrier inits visible too
  bool waited = !a.early || a.late;
  if (a.early && blockIdx.x == 0 && threadIdx.x == 0) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    waited = true;
  }
  // the merge grid that follows may be scheduled from now on (it waits for
  // this grid to finish before it reads anything)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int W = P.total;
  // Balanced ranges are dealt out transposed (range w = warp * gridDim.x + CTA):
  // neighbouring ranges -- often the same kind of work -- land on different
  // CTAs and SMs, so each SM gets a mix. Fixed splits keep the plain order.
  const int w = a.mode == kBalanced ? warp * (int)gridDim.x + (int)blockIdx.x
                                    : (int)blockIdx.x * NWARPS + warp;

  // Sequences with an empty context: out = 0, lse = -inf (balanced mode owns
  // them in CTA 0; fixed mode handles them through its empty partials).
  // (With split-K partitions, empty ones are skipped by the partition merge.)
  if (a.mode == kBalanced && parts == 1 && blockIdx.x == 0) {
    for (int pr = warp; pr < P.npairs; pr += NWARPS) {
      if (P.pair_off[pr + 1] != P.pair_off[pr]) continue;
      const int s = pr / parts;
      const int rslot = a.rows.slot;
      for (int h = 0; h < Hq; ++h) {
        const size_t row = (size_t)s * Hq + h;
        if (a.rows.o) {
          const size_t r = row * a.rows.stride + rslot;
          *reinterpret_cast<float4*>(a.rows.o + r * kHeadDim + lane * 4) =
              make_float4(0.f, 0.f, 0.f, 0.f);
          if (lane == 0) a.rows.lse[r] = neg_inf();
          continue;
        }
        *reinterpret_cast<uint2*>(a.out + row * kHeadDim + lane * 4) = make_uint2(0u, 0u);
        if (a.lse && lane == 0) a.lse[row] = neg_inf();
      }
    }
  }

  int R0 = 0, R1 = 0, fixed_p = 0;
  const int nw = min(a.num_workers, W);
  if (a.mode == kBalanced) {
    if (w < nw) {
      R0 = range_start(w, W, nw);
      R1 = range_start(w + 1, W, nw);
    }
  } else {
    const int PS = a.num_splits;
    if ((int64_t)w >= (int64_t)S * Hkv * PS) return;
    const int s = w / (Hkv * PS), h = (w / PS) % Hkv;
    fixed_p = w % PS;
    const int pr = P.seq_pair[s];
    const bool has = P.seq_pair[s + 1] > pr;
    const int nt = has ? (P.pair_off[pr + 1] - P.pair_off[pr]) / Hkv : 0;
    const int b0 = (int)((int64_t)fixed_p * nt / PS), b1 = (int)((int64_t)(fixed_p + 1) * nt / PS);
    if (b0 == b1) {
      // empty piece: P == 1 -> the row itself (0, -inf); else an empty partial
      for (int g = 0; g < kG; ++g) {
        const size_t row = (size_t)s * Hq + h * kG + g;
        if (PS == 1) {
          *reinterpret_cast<uint2*>(a.out + row * kHeadDim + lane * 4) = make_uint2(0u, 0u);
          if (a.lse && lane == 0) a.lse[row] = neg_inf();
        } else {
          *reinterpret_cast<float4*>(a.part_o + (row * PS + fixed_p) * kHeadDim + lane * 4) =
              make_float4(0.f, 0.f, 0.f, 0.f);
          if (lane == 0) a.part_lse[row * PS + fixed_p] = neg_inf();
        }
      }
      return;
    }
    R0 = P.pair_off[pr] + h * nt + b0;
    R1 = R0 + (b1 - b0);
  }
  if (R0 >= R1) {
    late_exit();
    return;
  }

  const int grp = lane >> 3;   // tokens 4*grp .. 4*grp+3 of a tile
  const int c8 = lane & 7;     // dims 16*c8 .. 16*c8+15
  const int hsel = lane & 1;   // head of the score this lane ends up holding

  // ---- producer state -----------------------------------------------------
  TilePos pp = locate(P, S, Hkv, R0);
  int pidx = R0;
  int wbase = R0;
  // block id of flat tile idx; tiles of a window lie a few pairs past pp
  // block of the sequence that tile t reads (its partition's first block + b)
  auto abs_block = [&](const TilePos& t) -> int {
    return parts > 1 ? t.b + part_begin(t.qt, (P.ctx[t.s] + kBlock - 1) / kBlock, parts) : t.b;
  };
  auto load_phys = [&](int idx) -> int {
    if (idx >= R1) return 0;
    const TilePos t = locate_from(P, Hkv, pp, idx);
    return a.block_tables[(size_t)t.s * a.max_blocks + abs_block(t)];
  };
  int phys_cur = load_phys(wbase + lane);
  int phys_next = load_phys(wbase + 32 + lane);

  auto issue = [&](int stage) {
    int phys = __shfl_sync(kFull, phys_cur, pidx - wbase);
    const bool first = (pidx == R0) || (pp.b == 0);
    if (lane == 0 && pidx != a.skip_copy) {
      if (phys < 0 || (int64_t)phys >= a.num_blocks) {
        flag_error(PA_DEVERR_BLOCK_RANGE);
        phys = 0;
      }
      if (!waited && pp.b == pp.nt - 1) {  // the tile that holds the new row
        asm volatile("griddepcontrol.wait;" ::: "memory");
        waited = true;
      }
      unsigned char* st = wbuf + stage * kStageBytes;
      const uint32_t bar = smem_addr(&bars[stage]);
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, F::kQOff + (first ? kQBytes : 0));
      const size_t tile = (size_t)phys * Hkv + pp.h;
      bulk_copy_g2s(smem_addr(st), a.k_cache + tile * F::kTile, F::kTile, bar);
      bulk_copy_g2s(smem_addr(st + F::kTile), a.v_cache + tile * F::kTile, F::kTile, bar);
      if (first)
        bulk_copy_g2s(smem_addr(st + F::kQOff),
                      a.q + ((size_t)pp.s * Hq + (size_t)pp.h * kG) * kHeadDim, kQBytes, bar);
    }
    ++pidx;
    if (pidx < R1) advance(P, S, Hkv, pp);
    if (pidx - wbase == 32) {
      wbase += 32;
      phys_cur = phys_next;
      phys_next = load_phys(wbase + 32 + lane);
    }
  };

  for (int i = 0; i < NSTAGE && pidx < R1; ++i) issue(i);

  // Waits for the copies of the k-th tile of this warp's range. false: a copy
  // never landed -- the remaining ones get a bounded wait and the warp stops.
  auto stage_ready = [&](int k) -> bool {
    if (mbar_wait_bounded(smem_addr(&bars[k % NSTAGE]), (uint32_t)(k / NSTAGE) & 1u)) return true;
    for (int j = k + 1; j < k + NSTAGE && R0 + j < pidx; ++j)
      mbar_wait_bounded(smem_addr(&bars[j % NSTAGE]), (uint32_t)(j / NSTAGE) & 1u);
    late_exit();
    return false;
  };

  // Writes one lane's 8 output dims (query head og of the tile's KV head,
  // dims od .. od+7, times inv) of a finished piece and, from lse_lane, its
  // log-sum-exp: the output row when the piece is a whole (sequence, KV head)
  // segment, else a partial -- the fixed split's slot, the partition's row or
  // the worker's slot -- for the merge.
  auto store_piece = [&](const TilePos& t, int og, int od, const float (&o8)[8], float inv,
                         float lse_own, bool lse_lane, bool complete, bool piece_first) {
    const size_t row = (size_t)t.s * Hq + (size_t)t.h * kG + og;
    if (a.mode == kFixed && a.num_splits > 1) {
      const int PS = a.num_splits;
      store_f8(a.part_o + (row * PS + fixed_p) * kHeadDim + od, o8, inv);
      if (lse_lane) a.part_lse[row * PS + fixed_p] = lse_own;
    } else if (complete && a.rows.o) {
      const size_t r = row * a.rows.stride + (parts > 1 ? t.qt : a.rows.slot);
      store_f8(a.rows.o + r * kHeadDim + od, o8, inv);
      if (lse_lane) a.rows.lse[r] = lse_own;
    } else if (complete) {
      store_out8(a.out + row * kHeadDim + od, o8, inv);
      if (a.lse && lse_lane) a.lse[row] = lse_own;
    } else {
      const size_t slot = (size_t)w * 2 + (piece_first ? 0 : 1);
      store_f8(a.part_o + (slot * kG + og) * kHeadDim + od, o8, inv);
      if (lse_lane) a.part_lse[slot * kG + og] = lse_own;
    }
  };

  if constexpr (Q8) {
    // ---- consumer, 8-bit tiles: the two contractions of a tile on warp MMAs
    // (m16n8k16, f16 operands, fp32 accumulation). Lane (g, c) = (lane / 4,
    // lane % 4). Scores: A = the K codes (rows = the tile's 16 tokens) as f16
    // (exact), B = q scaled by a power of two that puts its largest |q_d| in
    // [2^14, 2^15) (exact in f16: bf16 has 8 significant bits); column n of B
    // is head n & 1, so every lane ends with the scores of tokens g and g + 8
    // for both heads. The contraction order of the dims is free: for MMA j,
    // the k index pairs (2c, 2c+1) and (2c+8, 2c+9) are dims 32c + 4j + 0..3,
    // so each lane reads 32 contiguous bytes of rows g and g + 8.
    // Output: A = the V codes transposed (rows = dims, k = tokens), B = the
    // softmax weights times each row's V scale, divided by the largest such
    // product of the head in the tile (so in [0, 1], f16), and the MMA result
    // times that product joins the fp32 accumulator. For MMA m, row g is dim
    // 16g + 2m and row g + 8 is dim 16g + 2m + 1; k pairs (2c, 2c+1) and
    // (2c+8, 2c+9) are tokens 4c .. 4c+3, so each lane reads 16 contiguous
    // bytes of four token rows.
    const int g = lane >> 2, c = lane & 3;
    const int hq = g & 1;  // the head of B column g
    TilePos cp = locate(P, S, Hkv, R0);
    uint32_t qb[16];       // score B fragments: scaled q of head hq, f16 pairs
    float cq0 = 0.f, cq1 = 0.f;  // per head: scale_log2 / (power-of-two q scale)
    float acc[8][4];       // output accumulator, MMA C layout (see the finish)
    float m0 = neg_inf(), m1 = neg_inf(), l0 = 0.f, l1 = 0.f;
    int piece_b0 = 0;
    bool piece_first = true;
    float* pbuf = reinterpret_cast<float*>(wbuf + L::kPOff);

    int k = 0;
    for (int idx = R0; idx < R1; ++idx, ++k) {
      if (!stage_ready(k)) return;
      const int stage = k % NSTAGE;
      unsigned char* st = wbuf + stage * kStageBytes;
      const bool first = (idx == R0) || (cp.b == 0);
      if (first) {
        const uint4* qs = reinterpret_cast<const uint4*>(st + F::kQOff + hq * 256 + c * 64);
        float qv[32];
        float mx = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 u = qs[i];
          const uint32_t wq[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            qv[8 * i + 2 * j] = bf_lo(wq[j]);
            qv[8 * i + 2 * j + 1] = bf_hi(wq[j]);
            mx = fmaxf(mx, fmaxf(fabsf(qv[8 * i + 2 * j]), fabsf(qv[8 * i + 2 * j + 1])));
          }
        }
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
        // 2^(141 - e) for |q| max in [2^(e-127), 2^(e-126)); e >= 14 keeps it finite
        const int e = max((int)((__float_as_uint(mx) >> 23) & 0xffu), 14);
        const float qsc = __uint_as_float((uint32_t)(268 - e) << 23);
        const float cq = __fdiv_rn(a.scale_log2, qsc);
        const float cq_o = __shfl_xor_sync(kFull, cq, 4);  // lane g ^ 1: the other head
        cq0 = hq ? cq_o : cq;
        cq1 = hq ? cq : cq_o;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          qb[2 * j] = pack_h2(qv[4 * j] * qsc, qv[4 * j + 1] * qsc);
          qb[2 * j + 1] = pack_h2(qv[4 * j + 2] * qsc, qv[4 * j + 3] * qsc);
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
        m0 = neg_inf();
        m1 = neg_inf();
        l0 = 0.f;
        l1 = 0.f;
        piece_b0 = cp.b;
        piece_first = (idx == R0);
      }
      const int nvalid = min(kBlock, P.ctx[cp.s] - abs_block(cp) * kBlock);

      // ---- scores ---------------------------------------------------------------
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const uint4* kr0 = reinterpret_cast<const uint4*>(st + g * kHeadDim + c * 32);
        const uint4* kr1 = reinterpret_cast<const uint4*>(st + (g + 8) * kHeadDim + c * 32);
        const uint4 x0 = kr0[0], x1 = kr0[1], y0 = kr1[0], y1 = kr1[1];
        const uint32_t r0[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        const uint32_t r1[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
        float d2[4] = {0.f, 0.f, 0.f, 0.f};  // odd j: a second, independent chain
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t a0, a1, a2, a3;
          codes_to_h2<FMT>(r0[j], a0, a2);
          codes_to_h2<FMT>(r1[j], a1, a3);
          if (j & 1)
            mma_16816(d2, a0, a1, a2, a3, qb[2 * j], qb[2 * j + 1]);
          else
            mma_16816(d, a0, a1, a2, a3, qb[2 * j], qb[2 * j + 1]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) d[i] += d2[i];
      }
      const float* ksc = reinterpret_cast<const float*>(st + F::kScaleOff);
      const float kg0 = ksc[g], kg8 = ksc[g + 8];
      float s00 = d[0] * cq0 * kg0, s01 = d[1] * cq1 * kg0;  // token g, heads 0 / 1
      float s10 = d[2] * cq0 * kg8, s11 = d[3] * cq1 * kg8;  // token g + 8
      if (g >= nvalid) s00 = s01 = neg_inf();
      if (g + 8 >= nvalid) s10 = s11 = neg_inf();

      // ---- online softmax (log2 domain), per head over the 8 lane groups ---------
      float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      const float p00 = ex2(s00 - mn0), p01 = ex2(s01 - mn1);
      const float p10 = ex2(s10 - mn0), p11 = ex2(s11 - mn1);
      l0 = l0 * al0 + (p00 + p10);
      l1 = l1 * al1 + (p01 + p11);
      // weights [head][token] through shared memory to the lanes of B column g
      if (c < 2) {
        pbuf[g + 8 * c] = c ? p10 : p00;
        pbuf[16 + g + 8 * c] = c ? p11 : p01;
      }
      __syncwarp();
      const float4 pw = *reinterpret_cast<const float4*>(pbuf + hq * 16 + 4 * c);
      const float4 vs4 =
          *reinterpret_cast<const float4*>(st + F::kTile + F::kScaleOff + 16 * c);
      // weight x V scale of tokens 4c .. 4c+3 for head hq; rows past the
      // context may hold anything: their scale counts as 0
      const float x0 = pw.x * (4 * c < nvalid ? vs4.x : 0.f);
      const float x1 = pw.y * (4 * c + 1 < nvalid ? vs4.y : 0.f);
      const float x2 = pw.z * (4 * c + 2 < nvalid ? vs4.z : 0.f);
      const float x3 = pw.w * (4 * c + 3 < nvalid ? vs4.w : 0.f);
      // normalised by the head's largest in the tile: the weights that carry
      // the result keep f16's full relative precision, whatever the spread of
      // the rows' scales
      float xm = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
      xm = fmaxf(xm, __shfl_xor_sync(kFull, xm, 1));
      xm = fmaxf(xm, __shfl_xor_sync(kFull, xm, 2));
      const float rx = xm > 0.f ? 1.f / xm : 0.f;
      const float xm_o = __shfl_xor_sync(kFull, xm, 4);  // lane g ^ 1: the other head
      const float xm0 = hq ? xm_o : xm, xm1 = hq ? xm : xm_o;
      const uint32_t b0 = pack_h2(x0 * rx, x1 * rx);
      const uint32_t b1 = pack_h2(x2 * rx, x3 * rx);

      // ---- output ------------------------------------------------------------------
      const unsigned char* Vt = st + F::kTile;
      uint4 R[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        R[i] = *reinterpret_cast<const uint4*>(Vt + (4 * c + i) * kHeadDim + 16 * g);
      if constexpr (FMT == kFmtF8) {
        // E4M3 rows past the context may hold NaN codes: never let them into
        // the MMA (int8 codes are always finite and meet a zero weight)
        if (nvalid < kBlock) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (4 * c + i >= nvalid) R[i] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if (al0 != 1.f || al1 != 1.f) {
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          acc[m][0] *= al0;
          acc[m][1] *= al1;
          acc[m][2] *= al0;
          acc[m][3] *= al1;
        }
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int wd = m >> 1;
        // bytes (b, b+1) of each token row's word wd, interleaved by token
        const uint32_t sel = (m & 1) ? 0x7362u : 0x5140u;
        const uint32_t x01 = __byte_perm(word_of(R[0], wd), word_of(R[1], wd), sel);
        const uint32_t x23 = __byte_perm(word_of(R[2], wd), word_of(R[3], wd), sel);
        uint32_t a0, a1, a2, a3;
        codes_to_h2<FMT>(x01, a0, a1);
        codes_to_h2<FMT>(x23, a2, a3);
        float dv[4] = {0.f, 0.f, 0.f, 0.f};
        mma_16816(dv, a0, a1, a2, a3, b0, b1);
        acc[m][0] = fmaf(xm0, dv[0], acc[m][0]);
        acc[m][1] = fmaf(xm1, dv[1], acc[m][1]);
        acc[m][2] = fmaf(xm0, dv[2], acc[m][2]);
        acc[m][3] = fmaf(xm1, dv[3], acc[m][3]);
      }
      __syncwarp();  // all lanes are done with this stage and with pbuf
      if (pidx < R1) issue(stage);

      const bool last = (idx == R1 - 1) || (cp.b == cp.nt - 1);
      if (last) {
        // ---- finish the piece: acc[m] holds (dim 16g + 2m: head 0, head 1;
        // dim 16g + 2m + 1: head 0, head 1) in every lane of group g; lane
        // (g, c) writes head c >> 1, dims 16g + 8 (c & 1) .. +7 -------------------
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          l0 += __shfl_xor_sync(kFull, l0, o);
          l1 += __shfl_xor_sync(kFull, l1, o);
        }
        const int og = c >> 1;
        const bool hi = (c & 1) != 0;
        float o8[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float* lo_m = acc[i];
          const float* hi_m = acc[4 + i];
          const float e0 = hi ? hi_m[0] : lo_m[0], e1 = hi ? hi_m[1] : lo_m[1];
          const float e2 = hi ? hi_m[2] : lo_m[2], e3 = hi ? hi_m[3] : lo_m[3];
          o8[2 * i] = og ? e1 : e0;
          o8[2 * i + 1] = og ? e3 : e2;
        }
        const int od = 16 * g + (hi ? 8 : 0);
        const float lsum = og ? l1 : l0;
        const float lse_own = ((og ? m1 : m0) + lg2(lsum)) * kLn2;
        const float inv = 1.f / lsum;
        const bool complete = (piece_b0 == 0) && (cp.b == cp.nt - 1);
        const bool lse_lane = (lane & ~2) == 0;  // lanes 0 (head 0) and 2 (head 1)
        store_piece(cp, og, od, o8, inv, lse_own, lse_lane, complete, piece_first);
      }

      if (idx + 1 < R1) advance(P, S, Hkv, cp);
    }
  } else {
    constexpr int kRowB = 2 * kHeadDim;  // one bf16 token row, bytes
    // ---- consumer -------------------------------------------------------------
    // Lane (grp, c8) holds dims 16*c8..16*c8+15 of tokens 4*grp..4*grp+3 for
    // both query heads; fp32 pairs go through the packed (f32x2) FMA pipe.
    TilePos cp = locate(P, S, Hkv, R0);
    float2 q2[kG][8];    // scaled q, dims (16*c8 + 2j, +1)
    float2 acc[kG][8];   // output accumulator, same dims
    float m0 = neg_inf(), m1 = neg_inf(), l_lane = 0.f;
    int piece_b0 = 0;
    bool piece_first = true;

    int k = 0;
    for (int idx = R0; idx < R1; ++idx, ++k) {
      if (!stage_ready(k)) return;
      const int stage = k % NSTAGE;
      unsigned char* st = wbuf + stage * kStageBytes;
      const bool first = (idx == R0) || (cp.b == 0);
      if (first) {
#pragma unroll
        for (int g = 0; g < kG; ++g) {
          const uint4* qs = reinterpret_cast<const uint4*>(st + F::kQOff + g * 256 + c8 * 32);
          const uint4 qa = qs[0], qb = qs[1];
          const uint32_t wq[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            q2[g][j] = make_float2(bf_lo(wq[j]) * a.scale_log2, bf_hi(wq[j]) * a.scale_log2);
            acc[g][j] = make_float2(0.f, 0.f);
          }
        }
        m0 = neg_inf();
        m1 = neg_inf();
        l_lane = 0.f;
        piece_b0 = cp.b;
        piece_first = (idx == R0);
      }
      const int nvalid = min(kBlock, P.ctx[cp.s] - abs_block(cp) * kBlock);

      // ---- scores: 4 tokens x 2 heads of partial dots per lane ----------------
      float sc[8];
      const unsigned char* Ks = st + grp * 4 * kRowB + c8 * (kRowB / 8);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float2 kf[8];
        load_row16(Ks + i * kRowB, kf);
        float2 d0 = make_float2(0.f, 0.f), d1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          d0 = __ffma2_rn(q2[0][j], kf[j], d0);
          d1 = __ffma2_rn(q2[1][j], kf[j], d1);
        }
        sc[2 * i] = d0.x + d0.y;
        sc[2 * i + 1] = d1.x + d1.y;
      }
      // reduce-scatter over the 8 lanes of this group: value v = 2*i + g ends in
      // the lane with (lane & 7) == v
#pragma unroll
      for (int step = 0; step < 3; ++step) {
        const int half = 4 >> step;
        const bool upper = (lane & half) != 0;
#pragma unroll
        for (int j = 0; j < half; ++j) {
          const float send = upper ? sc[j] : sc[j + half];
          const float keep = upper ? sc[j + half] : sc[j];
          sc[j] = keep + __shfl_xor_sync(kFull, send, half);
        }
      }
      const int tok = grp * 4 + ((lane & 7) >> 1);
      const float s_val = tok < nvalid ? sc[0] : neg_inf();

      // ---- online softmax (log2 domain) ------------------------------------------
      float mx = s_val;
#pragma unroll
      for (int o = 2; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      const float mx_other = __shfl_xor_sync(kFull, mx, 1);
      const float mn0 = fmaxf(m0, hsel ? mx_other : mx);
      const float mn1 = fmaxf(m1, hsel ? mx : mx_other);
      const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      const float p = ex2(s_val - (hsel ? mn1 : mn0));
      l_lane = l_lane * (hsel ? al1 : al0) + p;
      float* pbuf = reinterpret_cast<float*>(wbuf + L::kPOff);
      pbuf[lane] = p;  // index 2*token + head
      __syncwarp();
      float pv[8];
      {
        const float4* pb = reinterpret_cast<const float4*>(pbuf + grp * 8);
        const float4 p0 = pb[0], p1 = pb[1];
        pv[0] = p0.x; pv[1] = p0.y; pv[2] = p0.z; pv[3] = p0.w;
        pv[4] = p1.x; pv[5] = p1.y; pv[6] = p1.z; pv[7] = p1.w;
      }
      if (al0 != 1.f || al1 != 1.f) {
        const float2 a0 = make_float2(al0, al0), a1 = make_float2(al1, al1);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          acc[0][j] = __fmul2_rn(acc[0][j], a0);
          acc[1][j] = __fmul2_rn(acc[1][j], a1);
        }
      }
      // ---- PV ----------------------------------------------------------------------
      const unsigned char* Vs = st + F::kTile + grp * 4 * kRowB + c8 * (kRowB / 8);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (nvalid == kBlock || grp * 4 + i < nvalid) {
          // tokens past the context may hold anything (even NaN): skip, never 0*x
          float2 vf[8];
          load_row16(Vs + i * kRowB, vf);
          const float2 p0 = make_float2(pv[2 * i], pv[2 * i]);
          const float2 p1 = make_float2(pv[2 * i + 1], pv[2 * i + 1]);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            acc[0][j] = __ffma2_rn(p0, vf[j], acc[0][j]);
            acc[1][j] = __ffma2_rn(p1, vf[j], acc[1][j]);
          }
        }
      }
      __syncwarp();  // all lanes are done with this stage's K/V and with pbuf
      // refill the stage now: finishing a piece below needs no stage memory, so
      // its work overlaps the copy
      if (pidx < R1) issue(stage);

      const bool last = (idx == R1 - 1) || (cp.b == cp.nt - 1);
      if (last) {
        // ---- finish the piece: sum the 4 token groups' accumulators (lanes
        // c8, c8+8, c8+16, c8+24) by a reduce-scatter over lane bits 4 and 3;
        // lane (b4, b3, c8) ends with head b4, dims 16*c8 + 8*b3 .. +7 ----------
        const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0;
        float h16[16];  // after lane bit 4: head b4, dims 16*c8 .. 16*c8+15
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float2 mine = b4 ? acc[1][j] : acc[0][j];
          const float2 send = b4 ? acc[0][j] : acc[1][j];
          h16[2 * j] = mine.x + __shfl_xor_sync(kFull, send.x, 16);
          h16[2 * j + 1] = mine.y + __shfl_xor_sync(kFull, send.y, 16);
        }
        float o8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float mine = b3 ? h16[8 + i] : h16[i];
          const float send = b3 ? h16[i] : h16[8 + i];
          o8[i] = mine + __shfl_xor_sync(kFull, send, 8);
        }
        float ls = l_lane;
#pragma unroll
        for (int o = 2; o < 32; o <<= 1) ls += __shfl_xor_sync(kFull, ls, o);
        const float lo = __shfl_xor_sync(kFull, ls, 1);
        const float l0 = hsel ? lo : ls, l1 = hsel ? ls : lo;
        const int og = b4 ? 1 : 0;             // output head of this lane
        const int od = c8 * 16 + (b3 ? 8 : 0);  // output dims od .. od+7
        const float lsum = og ? l1 : l0;
        const float lse_own = ((og ? m1 : m0) + lg2(lsum)) * kLn2;
        const float inv = 1.f / lsum;
        const bool complete = (piece_b0 == 0) && (cp.b == cp.nt - 1);
        const bool lse_lane = (lane & 15) == 0;
        store_piece(cp, og, od, o8, inv, lse_own, lse_lane, complete, piece_first);
      }

      if (idx + 1 < R1) advance(P, S, Hkv, cp);
    }
  }
  late_exit();
}

// Merge the pieces of every (sequence, KV head) that the balanced ranges cut.
// One warp per worker boundary. Launched as a dependent grid: while the decode
// grid still runs, each CTA rebuilds the same plan from context_lens (which
// the decode grid does not write) and each warp works out which segment it
// must merge; only then does it wait for the decode grid, so after the decode
// ends a single round of loads remains. Lane i reads piece i's lse values;
// the partial vectors of a round are loaded together.
__global__ void __launch_bounds__(256)
    decode_fixup_kernel(const int32_t* __restrict__ context_lens, int S, int Hkv, int max_blocks,
                        int num_workers, int parts, const float* __restrict__ part_o,
                        const float* __restrict__ part_lse, int Hq, uint16_t* __restrict__ out,
                        float* __restrict__ lse, const RowsOut rows) {
  // the next grid in the stream may start its own preparation now; it waits
  // for this grid before it reads anything this grid writes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ __align__(16) int fx_smem[];
  PlanSmem P;
  P.pair_off = fx_smem;
  P.seq_pair = P.pair_off + (S * parts + 1);
  P.ctx = P.seq_pair + (S + 1);
  P.qstart = P.ctx + S;
  PlanInputs in;
  in.context_lens = context_lens;
  in.cu_seqlens_q = nullptr;
  in.S = S;
  in.Hkv = Hkv;
  in.max_ctx = max_blocks * kBlock;
  in.qtile = 1;
  in.causal = 1;
  in.npairs_cap = S * parts;
  in.num_q_rows = S;
  in.parts = parts;
  build_plan(in, P, nullptr);
  const int W = P.total;
  const int nw = min(num_workers, W);
  const int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const MergeJob job = merge_job(P, S, Hkv, w, W, nw);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!job.valid) return;
  RowsOut r = rows;
  if (parts > 1) r.slot = job.qt;  // the partition's partial slot
  merge_segment(job, w, lane, part_o, part_lse, Hq, out, lse, r);
}

// Split-K merge over a regular [rows][heads][P][D] partial layout: one warp
// per (row, head).
__global__ void splitk_reduce_kernel(const float* __restrict__ part_o,
                                     const float* __restrict__ part_lse, int64_t nrh, int P,
                                     int D, uint16_t* __restrict__ out, float* __restrict__ lse) {
  const int64_t rh = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (rh >= nrh) return;
  const float* L = part_lse + rh * P;
  float mx = neg_inf();
  for (int i = lane; i < P; i += 32) mx = fmaxf(mx, L[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
  uint16_t* orow = out + rh * D;
  if (mx == neg_inf()) {
    for (int d = lane * 4; d < D; d += 128)
      *reinterpret_cast<uint2*>(orow + d) = make_uint2(0u, 0u);
    if (lse && lane == 0) lse[rh] = neg_inf();
    return;
  }
  float sum = 0.f;
  for (int i = lane; i < P; i += 32) sum += ex2((L[i] - mx) * kLog2e);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
  const float LSE = mx + lg2(sum) * kLn2;
  const float* O = part_o + rh * (int64_t)P * D;
  for (int d = lane * 4; d < D; d += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i0 = 0; i0 < P; i0 += 32) {
      const float wl = (i0 + lane < P) ? ex2((L[i0 + lane] - LSE) * kLog2e) : 0.f;
      const int n = min(32, P - i0);
      for (int j = 0; j < n; ++j) {
        const float wt = __shfl_sync(kFull, wl, j);
        const float4 o = *reinterpret_cast<const float4*>(O + (int64_t)(i0 + j) * D + d);
        acc.x = fmaf(wt, o.x, acc.x);
        acc.y = fmaf(wt, o.y, acc.y);
        acc.z = fmaf(wt, o.z, acc.z);
        acc.w = fmaf(wt, o.w, acc.w);
      }
    }
    uint2 o;
    o.x = pack_bf2(acc.x, acc.y);
    o.y = pack_bf2(acc.z, acc.w);
    *reinterpret_cast<uint2*>(orow + d) = o;
  }
  if (lse && lane == 0) lse[rh] = LSE;
}

// The split-K merge of decode partitions: the a7 formula over the [S][Hq][P]
// partials, where partition j of sequence s counts only if it holds blocks
// (part_begin(j) < part_begin(j + 1) for the sequence's context), so empty
// partitions are never written or read. A CTA has kPrWarps warps; RW of them
// share one (sequence, head) row: warp k of a row merges partitions k, k + RW,
// ... with the loads of a round of kMergeChunk partitions in flight together,
// then the row's warps combine their (max, sum, vector) through shared memory.
constexpr int kPrWarps = 8;

template <int RW>
__global__ void __launch_bounds__(kPrWarps * 32)
    parts_reduce_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                        const int32_t* __restrict__ context_lens, int max_ctx, int64_t nrh,
                        int Hq, int P, uint16_t* __restrict__ out, float* __restrict__ lse) {
  __shared__ float sm_m[kPrWarps], sm_l[kPrWarps];
  __shared__ float4 sm_acc[kPrWarps][32];
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int warp = wid % RW;  // warp within the row
  const int64_t rh = (int64_t)blockIdx.x * (kPrWarps / RW) + wid / RW;
  if (rh >= nrh) return;  // whole rows leave together (RW divides kPrWarps)
  const int s = (int)(rh / Hq);
  const int c = min(max(context_lens[s], 0), max_ctx);
  const int nt = (c + kBlock - 1) / kBlock;
  const float* L = part_lse + rh * P;
  const float* O = part_o + rh * (int64_t)P * kHeadDim;
  float mx = neg_inf(), sum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  // this warp's partitions: j = warp + RW * i
  const int mine = (P - warp + RW - 1) / RW;
  for (int i0 = 0; i0 < mine; i0 += kMergeChunk) {
    const int n = min(kMergeChunk, mine - i0);
    bool use[kMergeChunk];
    float li = neg_inf();
    float4 o[kMergeChunk];
#pragma unroll
    for (int k = 0; k < kMergeChunk; ++k) {
      const int j = warp + RW * (i0 + k);
      use[k] = k < n && part_begin(j, nt, P) < part_begin(j + 1, nt, P);
      o[k] = use[k] ? *reinterpret_cast<const float4*>(O + (int64_t)j * kHeadDim + lane * 4)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
      if (lane == k && use[k]) li = L[j];
    }
    float m = li;
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, x));
    m = fmaxf(m, mx);
    if (m == neg_inf()) continue;  // nothing in this round, nor before
    const float r = ex2((mx - m) * kLog2e);
    sum *= r;
    acc.x *= r; acc.y *= r; acc.z *= r; acc.w *= r;
    const float e = ex2((li - m) * kLog2e);  // weight of partition lane (0 if unused)
    float t = e;
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) t += __shfl_xor_sync(kFull, t, x);
    sum += t;
    mx = m;
#pragma unroll
    for (int k = 0; k < kMergeChunk; ++k) {
      const float wt = __shfl_sync(kFull, e, k);
      if (use[k]) {
        acc.x = fmaf(wt, o[k].x, acc.x);
        acc.y = fmaf(wt, o[k].y, acc.y);
        acc.z = fmaf(wt, o[k].z, acc.z);
        acc.w = fmaf(wt, o[k].w, acc.w);
      }
    }
  }
  if (RW > 1) {
    if (lane == 0) {
      sm_m[wid] = mx;
      sm_l[wid] = sum;
    }
    sm_acc[wid][lane] = acc;
    // the row's warps meet (a named barrier per row group)
    asm volatile("bar.sync %0, %1;" ::"r"(1 + wid / RW), "r"(RW * 32) : "memory");
    if (warp != 0) return;
  }
  const int w0 = wid;  // the row's first warp
  float M = neg_inf();
  if (RW > 1) {
#pragma unroll
    for (int k = 0; k < RW; ++k) M = fmaxf(M, sm_m[w0 + k]);
  } else {
    M = mx;
  }
  uint16_t* orow = out + rh * kHeadDim;
  if (M == neg_inf()) {  // every partition empty: an empty context
    *reinterpret_cast<uint2*>(orow + lane * 4) = make_uint2(0u, 0u);
    if (lse && lane == 0) lse[rh] = neg_inf();
    return;
  }
  float l = sum;
  float4 v = acc;
  if (RW > 1) {
    l = 0.f;
    v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < RW; ++k) {
      if (sm_m[w0 + k] == neg_inf()) continue;
      const float wk = ex2((sm_m[w0 + k] - M) * kLog2e);
      l = fmaf(wk, sm_l[w0 + k], l);
      const float4 ak = sm_acc[w0 + k][lane];
      v.x = fmaf(wk, ak.x, v.x);
      v.y = fmaf(wk, ak.y, v.y);
      v.z = fmaf(wk, ak.z, v.z);
      v.w = fmaf(wk, ak.w, v.w);
    }
  }
  const float inv = 1.f / l;
  uint2 ob;
  ob.x = pack_bf2(v.x * inv, v.y * inv);
  ob.y = pack_bf2(v.z * inv, v.w * inv);
  *reinterpret_cast<uint2*>(orow + lane * 4) = ob;
  if (lse && lane == 0) lse[rh] = M + lg2(l) * kLn2;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
constexpr int kWarps = 6;
// Batches with no more (sequence, KV head) segments than SMs (long contexts)
// run 8-warp CTAs, one per SM: each segment spans many warps and a sweep of
// CTA shapes measured the 8 x 32k batch 10% faster so; the other batches
// (engine, ragged) run best with 6 warps x 2 CTAs per SM.
constexpr int kWarpsLong = 8;
constexpr int kStages = 2;    // bf16: 2 x 8 KB of copies in flight per warp
// 8-bit pools (int8, FP8): 8 warps x 2 stages of 4.7 KB (a K and a V tile,
// each one copy of codes and scales), two CTAs per SM. Resident warps pay
// more than stages: 16 per SM measured 6-11% faster than 12 (6 x 2) on the
// ragged and long batches, while 7 x 3, 6 x 3 and 5 x 4 stages were 4-25%
// slower; 3 CTAs of 6 warps need under 113 registers and spill. With the
// per-tile math taken out, the 8 x 32k batch still takes 97% of its time:
// there the 2112-byte copies, not the MMA loop, set the pace.
constexpr int kWarpsQ8 = 8;
constexpr int kStagesQ8 = 2;

struct DecodeGeometry;
using DecodeLaunch = cudaError_t (*)(const DecodeGeometry&, const DecodeArgs&, cudaStream_t);

struct DecodeGeometry {
  DecodeLaunch launch = nullptr;  // the decode grid of this shape
  int mode = kBalanced;
  int P = 0;
  int grid = 0;
  int workers = 0;
  size_t smem = 0;
  size_t fixup_smem = 0;
  size_t ws_desc = 0, ws_lse = 0, ws_o = 0, ws_plse = 0, ws_po = 0, ws_bytes = 0;
  int parts = 1;  // balanced: split-K partitions per sequence
  int nwarps = kWarps;  // warps per CTA of the decode grid
  int nstages = kStages;  // stages per warp
};

// A CTA shape of the decode grid: NW warps of NST stages, pool format FMT.
template <int FMT, int NW, int NST>
struct DecodeShape {
  static cudaError_t launch(const DecodeGeometry& g, const DecodeArgs& a, cudaStream_t st) {
    return launch_dependent(paged_decode_kernel<NW, NST, FMT>, dim3(g.grid), dim3(NW * 32), g.smem,
                            st, a);
  }
};

// shared memory of the plan: pair_off [S * parts + 1], seq_pair [S + 1], ctx [S],
// qstart [S + 1], and 40 spare ints
inline size_t plan_smem_bytes(int S, int parts = 1) {
  return sizeof(int) * ((size_t)S * parts + 1 + 3 * (size_t)S + 2 + 40);
}

// max_sms > 0: size the balanced grid for that many SMs (the rest are busy).
// num_splits 0: balanced cut of the sequences' tiles; P >= 2: balanced cut of
// the tiles of P partitions per sequence when their plan fits in shared
// memory (the kFixed layout of one warp per partition otherwise); 1: kFixed.
template <int FMT, int NW, int NST>
int decode_geometry_t(const pa_shape* sh, int num_splits, DecodeGeometry* g, int max_sms = 0) {
  constexpr int kWarps = NW;
  g->nwarps = NW;
  g->nstages = NST;
  g->launch = &DecodeShape<FMT, NW, NST>::launch;
  DeviceInfo dev;
  if (!current_device_info(&dev)) return PA_ERR_CUDA;
  const int S = sh->num_seqs, Hkv = sh->num_kv_heads, Hq = sh->num_q_heads;
  const void* kern = reinterpret_cast<const void*>(paged_decode_kernel<NW, NST, FMT>);
  if (!raise_smem_limit(kern)) return PA_ERR_CUDA;
  const size_t warp_bytes = (size_t)kWarps * WarpLayout<NST, FMT>::kBytes;
  const int parts = num_splits >= 2 ? num_splits : 1;
  if (num_splits != 1 && warp_bytes + plan_smem_bytes(S, parts) <= (size_t)dev.max_smem_optin) {
    g->smem = warp_bytes + plan_smem_bytes(S, parts);
    int per_sm = 0;
    if (!kernel_occupancy(kern, kWarps * 32, g->smem, &per_sm) || per_sm <= 0)
      return PA_ERR_CUDA;
    g->mode = kBalanced;
    g->parts = parts;
    g->P = num_splits;
    g->grid = (max_sms > 0 && max_sms < dev.num_sms ? max_sms : dev.num_sms) * per_sm;
    g->workers = g->grid * kWarps;
    g->fixup_smem = plan_smem_bytes(S, parts);
    if (g->fixup_smem > (size_t)dev.max_smem_optin) return PA_ERR_UNSUPPORTED;
    if (g->fixup_smem > 48 * 1024 &&
        !raise_smem_limit(reinterpret_cast<const void*>(decode_fixup_kernel)))
      return PA_ERR_CUDA;
    g->ws_lse = round_up(sizeof(float) * 2 * kG * (size_t)g->workers, 256);
    g->ws_o = round_up(sizeof(float) * 2 * kG * kHeadDim * (size_t)g->workers, 256);
    if (parts > 1) {  // the partitions' partials, merged by pa_splitk_reduce
      g->ws_plse = round_up(sizeof(float) * (size_t)S * Hq * parts, 256);
      g->ws_po = round_up(sizeof(float) * (size_t)S * Hq * parts * kHeadDim, 256);
    }
  } else {
    g->smem = warp_bytes + plan_smem_bytes(S);
    if (g->smem > (size_t)dev.max_smem_optin) return PA_ERR_UNSUPPORTED;
    g->mode = kFixed;
    g->P = num_splits;
    const int64_t warps = (int64_t)S * Hkv * num_splits;
    if ((warps + kWarps - 1) / kWarps > 0x7fffffff) return PA_ERR_ARG;
    g->grid = (int)((warps + kWarps - 1) / kWarps);
    g->workers = (int)warps;
    if (num_splits > 1) {
      g->ws_lse = round_up(sizeof(float) * (size_t)S * Hq * num_splits, 256);
      g->ws_o = round_up(sizeof(float) * (size_t)S * Hq * num_splits * kHeadDim, 256);
    }
  }
  g->ws_bytes = g->ws_desc + g->ws_lse + g->ws_o + g->ws_plse + g->ws_po;
  return PA_OK;
}

int decode_geometry(const pa_shape* sh, int num_splits, DecodeGeometry* g, int fmt = kFmtBf16,
                    int max_sms = 0) {
  if (fmt == kFmtI8)
    return decode_geometry_t<kFmtI8, kWarpsQ8, kStagesQ8>(sh, num_splits, g, max_sms);
  if (fmt == kFmtF8)
    return decode_geometry_t<kFmtF8, kWarpsQ8, kStagesQ8>(sh, num_splits, g, max_sms);
  DeviceInfo dev;
  if (!current_device_info(&dev)) return PA_ERR_CUDA;
  const bool long_ctx = num_splits != 1 && max_sms == 0 &&
                        (int64_t)sh->num_seqs * sh->num_kv_heads <= dev.num_sms;
  return long_ctx ? decode_geometry_t<kFmtBf16, kWarpsLong, kStages>(sh, num_splits, g, max_sms)
                  : decode_geometry_t<kFmtBf16, kWarps, kStages>(sh, num_splits, g, max_sms);
}

int check_decode_args(const pa_shape* shape, int num_splits) {
  int rc = check_shape_common(shape);
  if (rc != PA_OK) return rc;
  if (shape->num_q_heads != kG * shape->num_kv_heads) return PA_ERR_UNSUPPORTED;
  if (num_splits < 0 || num_splits > 1024) return PA_ERR_ARG;
  if ((int64_t)shape->num_seqs * shape->num_kv_heads * (shape->max_blocks_per_seq + 1) >
      0x3fffffff)
    return PA_ERR_ARG;
  return PA_OK;
}

}  // namespace

unsigned take_error_word_decode(cudaStream_t stream, int* rc) {
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

using namespace pa;

extern "C" size_t pa_decode_workspace_size(const pa_shape* shape, int num_splits) {
  if (check_decode_args(shape, num_splits) != PA_OK) return 0;
  if (shape->num_seqs == 0) return 0;
  DecodeGeometry g;
  if (decode_geometry(shape, num_splits, &g) != PA_OK) return 0;
  return g.ws_bytes;
}

extern "C" size_t pa_decode_int8_workspace_size(const pa_shape* shape, int num_splits) {
  if (check_decode_args(shape, num_splits) != PA_OK) return 0;
  if (shape->num_seqs == 0) return 0;
  DecodeGeometry g;
  if (decode_geometry(shape, num_splits, &g, kFmtI8) != PA_OK) return 0;
  return g.ws_bytes;
}

extern "C" size_t pa_decode_fp8_workspace_size(const pa_shape* shape, int num_splits) {
  if (check_decode_args(shape, num_splits) != PA_OK) return 0;
  if (shape->num_seqs == 0) return 0;
  DecodeGeometry g;
  if (decode_geometry(shape, num_splits, &g, kFmtF8) != PA_OK) return 0;
  return g.ws_bytes;
}

namespace pa {
namespace {

// Failure-detection hook (pa_debug_inject_missing_copy): consumed by the next
// decode launch of this host thread.
thread_local int g_inject_missing_copy = -1;

// Validate, size and launch the decode grid and its merge. `early`: see the
// kernel (only pa_append_decode sets it).
// fmt selects the pool format (bf16, int8 or FP8 tiles).
int decode_impl(const pa_bf16* q, const void* k_cache, const void* v_cache, int fmt,
                const int32_t* block_tables, const int32_t* context_lens, float scale,
                pa_bf16* out, float* lse, const pa_shape* shape, int num_splits,
                void* workspace, size_t workspace_bytes, cudaStream_t st, int early,
                const RowsOut* rows = nullptr, int late = 0, int max_sms = 0) {
  int rc = check_decode_args(shape, num_splits);
  if (rc != PA_OK) return rc;
  if (shape->num_seqs == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || (!out && !rows))
    return PA_ERR_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4) || (lse && !aligned(lse, 4)))
    return PA_ERR_ARG;
  if (!(scale == scale)) return PA_ERR_ARG;
  DecodeGeometry g;
  rc = decode_geometry(shape, num_splits, &g, fmt, max_sms);
  if (rc != PA_OK) return rc;
  if (g.ws_bytes > 0 &&
      (!workspace || workspace_bytes < g.ws_bytes || !aligned(workspace, 256)))
    return PA_ERR_WORKSPACE;

  DecodeArgs a;
  a.q = q;
  a.k_cache = static_cast<const unsigned char*>(k_cache);
  a.v_cache = static_cast<const unsigned char*>(v_cache);
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.out = out;
  a.lse = lse;
  a.scale_log2 = (float)((double)scale * 1.4426950408889634);
  a.S = shape->num_seqs;
  a.Hq = shape->num_q_heads;
  a.Hkv = shape->num_kv_heads;
  a.max_blocks = shape->max_blocks_per_seq;
  a.num_blocks = shape->num_blocks;
  a.mode = g.mode;
  a.num_splits = g.P;
  a.num_workers = g.workers;
  a.parts = g.parts;
  a.early = early;
  a.late = late;
  if (late && (early || g.mode != kBalanced)) return PA_ERR_ARG;
  a.skip_copy = g_inject_missing_copy;
  g_inject_missing_copy = -1;
  if (rows) {
    if (g.mode != kBalanced || g.parts > 1 || !rows->o || !rows->lse) return PA_ERR_ARG;
    a.rows = *rows;
  }
  char* ws = static_cast<char*>(workspace);
  a.part_lse = g.ws_lse ? reinterpret_cast<float*>(ws + g.ws_desc) : nullptr;
  a.part_o = g.ws_o ? reinterpret_cast<float*>(ws + g.ws_desc + g.ws_lse) : nullptr;
  float* plse = nullptr;
  float* po = nullptr;
  if (g.parts > 1) {
    // finished partitions land as fp32 partials [S][Hq][P], slot = partition
    plse = reinterpret_cast<float*>(ws + g.ws_desc + g.ws_lse + g.ws_o);
    po = reinterpret_cast<float*>(ws + g.ws_desc + g.ws_lse + g.ws_o + g.ws_plse);
    a.rows.o = po;
    a.rows.lse = plse;
    a.rows.stride = g.parts;
    a.rows.slot = 0;
    a.rows.tokens = a.S;
  }

  if (g.launch(g, a, st) != cudaSuccess) return PA_ERR_CUDA;
  const int wpb = 8;
  if (g.mode == kBalanced) {
    // the merge grid may be scheduled while the decode grid drains; it waits
    // for the decode grid's completion before reading
    if (launch_dependent(decode_fixup_kernel, dim3((g.workers + wpb - 1) / wpb), dim3(wpb * 32),
                         g.fixup_smem, st, context_lens, a.S, a.Hkv, a.max_blocks, g.workers,
                         g.parts, (const float*)a.part_o, (const float*)a.part_lse, a.Hq,
                         (uint16_t*)out, lse, a.rows) != cudaSuccess)
      return PA_ERR_CUDA;
    if (g.parts > 1) {  // the split-K merge of the P partitions
      const int64_t nrh = (int64_t)a.S * a.Hq;
      // warps per row: one round of up to 8 partitions each
      const int rw = g.parts >= 64 ? 8 : g.parts >= 32 ? 4 : g.parts >= 16 ? 2 : 1;
      const unsigned blocks = (unsigned)((nrh * rw + kPrWarps - 1) / kPrWarps);
      const int mctx = a.max_blocks * kBlock;
      if (rw == 8)
        parts_reduce_kernel<8><<<blocks, kPrWarps * 32, 0, st>>>(po, plse, context_lens, mctx,
                                                                  nrh, a.Hq, g.parts, out, lse);
      else if (rw == 4)
        parts_reduce_kernel<4><<<blocks, kPrWarps * 32, 0, st>>>(po, plse, context_lens, mctx,
                                                                  nrh, a.Hq, g.parts, out, lse);
      else if (rw == 2)
        parts_reduce_kernel<2><<<blocks, kPrWarps * 32, 0, st>>>(po, plse, context_lens, mctx,
                                                                  nrh, a.Hq, g.parts, out, lse);
      else
        parts_reduce_kernel<1><<<blocks, kPrWarps * 32, 0, st>>>(po, plse, context_lens, mctx,
                                                                  nrh, a.Hq, g.parts, out, lse);
    }
  } else if (g.P > 1) {
    const int64_t nrh = (int64_t)a.S * a.Hq;
    splitk_reduce_kernel<<<(unsigned)((nrh + wpb - 1) / wpb), wpb * 32, 0, st>>>(
        a.part_o, a.part_lse, nrh, g.P, kHeadDim, out, lse);
  }
  if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

}  // namespace

int decode_rows(const pa_bf16* q, const pa_bf16* k_cache, const pa_bf16* v_cache,
                const int32_t* block_tables, const int32_t* context_lens, float scale,
                const pa_shape* shape, const RowsOut& rows, void* workspace,
                size_t workspace_bytes, cudaStream_t st, int late, int max_sms) {
  return decode_impl(q, k_cache, v_cache, kFmtBf16, block_tables, context_lens, scale,
                     nullptr, nullptr, shape, 0, workspace, workspace_bytes, st, 0, &rows, late,
                     max_sms);
}

size_t decode_rows_workspace_size(const pa_shape* shape, int max_sms) {
  if (check_decode_args(shape, 0) != PA_OK || shape->num_seqs == 0) return 0;
  DecodeGeometry g;
  if (decode_geometry(shape, 0, &g, kFmtBf16, max_sms) != PA_OK) return 0;
  return g.ws_bytes;
}

}  // namespace pa

extern "C" int pa_decode(const pa_bf16* q, const pa_bf16* k_cache, const pa_bf16* v_cache,
                         const int32_t* block_tables, const int32_t* context_lens, float scale,
                         pa_bf16* out, float* lse, const pa_shape* shape, int num_splits,
                         void* workspace, size_t workspace_bytes, void* stream) {
  pa::NvtxRange nvtx_range("pa_decode");
  return decode_impl(q, k_cache, v_cache, kFmtBf16, block_tables, context_lens, scale,
                     out, lse, shape, num_splits, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream), 0);
}

extern "C" int pa_decode_int8(const pa_bf16* q, const uint8_t* k_cache, const uint8_t* v_cache,
                              const int32_t* block_tables, const int32_t* context_lens,
                              float scale, pa_bf16* out, float* lse, const pa_shape* shape,
                              int num_splits, void* workspace, size_t workspace_bytes,
                              void* stream) {
  pa::NvtxRange nvtx_range("pa_decode_int8");
  return decode_impl(q, k_cache, v_cache, kFmtI8, block_tables, context_lens, scale, out, lse,
                     shape, num_splits, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream), 0);
}

extern "C" int pa_decode_fp8(const pa_bf16* q, const uint8_t* k_cache, const uint8_t* v_cache,
                             const int32_t* block_tables, const int32_t* context_lens,
                             float scale, pa_bf16* out, float* lse, const pa_shape* shape,
                             int num_splits, void* workspace, size_t workspace_bytes,
                             void* stream) {
  pa::NvtxRange nvtx_range("pa_decode_fp8");
  return decode_impl(q, k_cache, v_cache, kFmtF8, block_tables, context_lens, scale, out, lse,
                     shape, num_splits, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream), 0);
}

extern "C" int pa_append_decode(const pa_bf16* k_new, const pa_bf16* v_new,
                                const int64_t* slot_mapping, int64_t num_new_tokens,
                                const pa_bf16* q, pa_bf16* k_cache, pa_bf16* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens,
                                float scale, pa_bf16* out, float* lse, const pa_shape* shape,
                                void* workspace, size_t workspace_bytes, void* stream) {
  pa::NvtxRange nvtx_range("pa_append_decode");
  // check everything first so that a failing call enqueues nothing
  int rc = check_decode_args(shape, 0);
  if (rc != PA_OK) return rc;
  if (num_new_tokens < 0) return PA_ERR_ARG;
  if (num_new_tokens > 0 &&
      (!k_new || !v_new || !slot_mapping || !aligned(k_new, 16) || !aligned(v_new, 16) ||
       !aligned(slot_mapping, 8)))
    return PA_ERR_ARG;
  if (shape->num_seqs > 0) {
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PA_ERR_ARG;
    DecodeGeometry g;
    rc = decode_geometry(shape, 0, &g);
    if (rc != PA_OK) return rc;
    if (!workspace || workspace_bytes < g.ws_bytes || !aligned(workspace, 256))
      return PA_ERR_WORKSPACE;
  }
  rc = pa_reshape_and_cache(k_new, v_new, slot_mapping, num_new_tokens, k_cache, v_cache, shape,
                            stream);
  if (rc != PA_OK) return rc;
  // with new tokens, the cache write ran just before: the decode prologue
  // (which reads only context_lens and block_tables) and every tile but the
  // segments' last ones may overlap it
  return decode_impl(q, k_cache, v_cache, kFmtBf16, block_tables, context_lens, scale,
                     out, lse, shape, 0, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream), num_new_tokens > 0 ? 1 : 0);
}

extern "C" int pa_splitk_reduce(const float* part_out, const float* part_lse, int64_t num_rows,
                                int num_heads, int num_splits, int head_dim, pa_bf16* out,
                                float* lse, void* stream) {
  pa::NvtxRange nvtx_range("pa_splitk_reduce");
  if (num_rows < 0 || num_heads <= 0 || num_splits <= 0 || head_dim <= 0) return PA_ERR_ARG;
  if (head_dim % 4 != 0 || head_dim > 1024) return PA_ERR_UNSUPPORTED;
  if (num_rows == 0) return PA_OK;
  if (!part_out || !part_lse || !out) return PA_ERR_ARG;
  if (!aligned(part_out, 16) || !aligned(part_lse, 4) || !aligned(out, 8) ||
      (lse && !aligned(lse, 4)))
    return PA_ERR_ARG;
  const int64_t nrh = num_rows * num_heads;
  const int wpb = 8;
  const int64_t blocks = (nrh + wpb - 1) / wpb;
  if (blocks > 0x7fffffff) return PA_ERR_ARG;
  splitk_reduce_kernel<<<(unsigned)blocks, wpb * 32, 0, static_cast<cudaStream_t>(stream)>>>(
      part_out, part_lse, nrh, num_splits, head_dim, out, lse);
  if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

// ---------------------------------------------------------------------------
// pa_decode_static_scratch: pa_decode (balanced split) for callers that are
// not allowed to allocate device memory themselves -- for example a plugin
// running inside another runtime that owns every device allocation, or a
// serving loop whose memory is planned once up front, where a cudaMalloc would
// also synchronise the device. Its split scratch is this file-scope array
// instead of a caller workspace. The array is part of the library image: every
// GPU that loads the library holds these bytes until the process exits.
// ---------------------------------------------------------------------------
namespace pa {
namespace {

// 8 MiB. The balanced split needs 2 partial slots x 2 heads x 129 fp32 per
// resident warp: 3.6 MiB on a 152-SM GB300 (1824 warps), so the array covers
// devices of up to about 300 SMs at this CTA shape.
constexpr size_t kStaticScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_pa_static_scratch[kStaticScratchBytes];

// Device address of the scratch array in the current context. In host code the
// array's name is only a host-side stand-in, so the real address is looked up
// (cudaGetSymbolAddress, with the device current) the first time a context
// calls, and cached per context: a new context on the same device (after a
// device reset, for instance) looks it up again.
void* static_scratch_address(int* rc) {
  using GetCtx = CUresult (*)(CUcontext*);
  static GetCtx get_ctx = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_ctx = reinterpret_cast<GetCtx>(p);
  });
  if (get_ctx == nullptr) {
    *rc = PA_ERR_CUDA;
    return nullptr;
  }
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) == CUDA_SUCCESS && ctx == nullptr) {
    // no context on this thread yet: the runtime creates the device's primary
    // context at its first call that needs one
    if (cudaFree(nullptr) != cudaSuccess) {
      *rc = PA_ERR_CUDA;
      return nullptr;
    }
    get_ctx(&ctx);
  }
  if (ctx == nullptr) {
    *rc = PA_ERR_CUDA;
    return nullptr;
  }
  static std::mutex mu;
  static std::map<CUcontext, void*> addr;
  std::lock_guard<std::mutex> lock(mu);
  const auto it = addr.find(ctx);
  if (it != addr.end()) return it->second;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_pa_static_scratch) != cudaSuccess || p == nullptr) {
    *rc = PA_ERR_CUDA;
    return nullptr;
  }
  addr[ctx] = p;
  return p;
}

}  // namespace
}  // namespace pa

extern "C" int pa_decode_static_scratch(const pa_bf16* q, const pa_bf16* k_cache,
                                        const pa_bf16* v_cache, const int32_t* block_tables,
                                        const int32_t* context_lens, float scale, pa_bf16* out,
                                        float* lse, const pa_shape* shape, void* stream) {
  pa::NvtxRange nvtx_range("pa_decode_static_scratch");
  int rc = check_decode_args(shape, 0);
  if (rc != PA_OK) return rc;
  if (shape->num_seqs == 0) return PA_OK;
  DecodeGeometry g;
  rc = decode_geometry(shape, 0, &g);
  if (rc != PA_OK) return rc;
  if (g.ws_bytes > kStaticScratchBytes) return PA_ERR_WORKSPACE;  // beyond the fixed array
  rc = PA_OK;
  void* scratch = static_scratch_address(&rc);
  if (scratch == nullptr) return rc;
  return pa_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, lse, shape, 0,
                   scratch, kStaticScratchBytes, stream);
}

extern "C" int pa_debug_inject_missing_copy(int flat_tile) {
  pa::g_inject_missing_copy = flat_tile < 0 ? -1 : flat_tile;
  return PA_OK;
}
