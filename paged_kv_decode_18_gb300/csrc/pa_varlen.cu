// pa_varlen.cu -- paged attention for several query tokens per sequence:
// speculative-decoding verify (1 + k draft tokens, causal inside the query
// window) and chunked prefill (a chunk of queries at an offset whose earlier
// tokens are already cached), over the same block pool as decode.
//
// Pages: "S20 - The Complete Engine", section "Core idea" (step 3 PROPOSE
// attaches draft tokens, step 5 verifies them in the same forward); course
// README "Build an LLM Inference Engine From Scratch", curriculum rows
// "Batching & Scheduling" (chunked prefill, FlashAttention) and "Decoding
// Acceleration" (speculative decoding), and its claim that online softmax is
// exact and split-K variants agree.
//
// Query j of a sequence with q_len Lq and context c sits at position
// c - Lq + j and (causal) sees keys 0 .. c - Lq + j.
//
// Design (GB300): q_len x group rows per KV head make QK^T and PV real
// matrix products, so they run on the tensor cores (mma.sync m16n8k16, bf16
// in, fp32 accumulate) in tiles of 16 rows = (16/G) query tokens x G query
// heads of one KV head against 16-key blocks:
//   * K/V tiles arrive by 2-D TMA (cp.async.bulk.tensor) with the 128-byte
//     swizzle, so ldmatrix reads them without bank conflicts; each warp loads
//     the Q fragments of a (sequence, query tile) straight into registers when
//     it starts one (a stage is only the 8 KB K/V tile);
//   * one warp is one worker with a private ring of stages and a contiguous
//     range of the batch's (sequence, query tile, KV head, block) tiles -- the
//     same equal-range balancing as decode, so verify sequences, prefill
//     chunks and ragged lengths spread evenly over the GPU;
//   * online softmax on the accumulator fragments, P rounded to bf16 for the
//     PV product (as FlashAttention does), running sums kept in fp32.
#include <cudaTypedefs.h>

#include "pa_device.cuh"
#include "pa_host.h"

namespace pa {
namespace {

constexpr int kRows = 16;                      // rows of one query tile
constexpr int kHalfBytes = kBlock * 128;       // 16 rows x 128 B (64 dims), swizzled
constexpr int kStageBytes = 4 * kHalfBytes;  // K0 K1 V0 V1 = 8 KB
constexpr int kDescInts = 8;

struct VarlenArgs {
  const uint16_t* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* cu_seqlens_q;
  uint16_t* out;
  float* lse;
  float scale_log2;
  int S, Hq, Hkv, G, QT, max_blocks;
  int64_t num_blocks;
  int64_t num_q_tokens;
  int causal;
  int npairs_cap;
  int num_workers;
  int max_lq;       // longer sequences go to the tcgen05 prefill kernel
  float* part_o;    // [NW*2][16][D]
  float* part_lse;  // [NW*2][16]
  int* desc;        // [NW][kDescInts]
  // 1: the grid ahead (the tcgen05 prefill grid of the same call, which
  // waited for its own predecessor before letting this grid launch) is not
  // waited for before the work: this grid reads nothing it writes and writes
  // nothing it reads, so verify tiles stream on the SMs that the prefill
  // grid's tail leaves free
  int late;
  // > 0 (with late): the prefill grid ahead runs beside this one on K of its
  // `split` CTAs (overlap_split); this grid works on the other SMs' share of
  // its CTAs, the first ones launched
  int split;
};

// byte offset of (row, 16-byte chunk) inside a 16 x 128 B box written by TMA
// with the 128-byte swizzle (chunk index XOR row mod 8)
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <int NWARPS, int NSTAGE>
__device__ __forceinline__ void varlen_body(const CUtensorMap& tmk, const CUtensorMap& tmv,
                                            const VarlenArgs& a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // stage buffers need 1024-byte alignment for the swizzle pattern
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned char* wbuf = smem + warp * (NSTAGE * kStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NWARPS * NSTAGE * kStageBytes) +
                   warp * NSTAGE;
  const int S = a.S, Hkv = a.Hkv, Hq = a.Hq, G = a.G, QT = a.QT;

  int* pm = reinterpret_cast<int*>(smem + NWARPS * NSTAGE * kStageBytes + NWARPS * NSTAGE * 8);
  PlanSmem P;
  P.pair_off = pm;
  P.seq_pair = P.pair_off + (a.npairs_cap + 1);
  P.ctx = P.seq_pair + (S + 1);
  P.qstart = P.ctx + S;
  int* scratch = P.qstart + (S + 1);

  if (lane == 0) {
    for (int i = 0; i < NSTAGE; ++i) mbar_init(smem_addr(&bars[i]), 1);
    mbar_fence_init();
  }
  if (threadIdx.x == 0) {
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  // launched as a programmatic dependent of the previous grid: wait for it
  // before reading anything it may have written (late: see VarlenArgs)
  if (!a.late) asm volatile("griddepcontrol.wait;" ::: "memory");
  PlanInputs in;
  in.context_lens = a.context_lens;
  in.cu_seqlens_q = a.cu_seqlens_q;
  in.S = S;
  in.Hkv = Hkv;
  in.max_ctx = a.max_blocks * kBlock;
  in.qtile = QT;
  in.causal = a.causal;
  in.npairs_cap = a.npairs_cap;
  in.num_q_rows = a.num_q_tokens;
  in.max_lq = a.max_lq;
  build_plan(in, P, scratch);
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int W = P.total;
  // CTAs that take work: all, or beside a prefill grid that keeps K of N
  // SMs, the share of the other N - K (the CTAs launched first)
  int ctas = (int)gridDim.x;
  if (a.split > 0) {
    const uintptr_t r = reinterpret_cast<uintptr_t>(scratch);
    const int K = overlap_split(a.cu_seqlens_q, a.context_lens, S, Hkv, G, a.causal,
                                a.max_lq + 1, a.max_blocks * kBlock, a.split,
                                reinterpret_cast<unsigned long long*>((r + 7) & ~uintptr_t(7)));
    ctas = max(1, (int)(((int64_t)gridDim.x * (a.split - K)) / a.split));
  }
  // ranges are dealt out transposed (range w = warp * ctas + CTA):
  // neighbouring ranges -- often the same kind of work -- land on different
  // CTAs and SMs, so each SM gets a mix; the CTAs past `ctas` hold the
  // remaining (empty) worker slots
  const int w = (int)blockIdx.x < ctas
                    ? warp * ctas + (int)blockIdx.x
                    : ctas * NWARPS + ((int)blockIdx.x - ctas) * NWARPS + warp;
  const int nw = min(ctas * NWARPS, W);
  int R0 = 0, R1 = 0;
  if (w < nw) {
    R0 = (int)((int64_t)w * W / nw);
    R1 = (int)((int64_t)(w + 1) * W / nw);
  }
  if (w < a.num_workers && lane == 0) {
    int d[5] = {-1, 0, 0, 0, 0};
    if (R0 < R1) {
      const TilePos t = locate(P, S, Hkv, R0);
      const int A = R0 - t.b;
      const int R0prev = w > 0 ? (int)((int64_t)(w - 1) * W / nw) : 0;
      if (t.b > 0 && A >= R0prev) {
        d[0] = t.s;
        d[1] = t.qt;
        d[2] = t.h;
        d[3] = (int)(((int64_t)(A + t.nt) * nw - 1) / W);
        d[4] = (A == R0prev) ? 0 : 1;
      }
    }
    int* dd = a.desc + (size_t)w * kDescInts;
    for (int i = 0; i < 5; ++i) dd[i] = d[i];
  }
  if (R0 >= R1) return;

  // ---- producer --------------------------------------------------------------
  TilePos pp = locate(P, S, Hkv, R0);
  int pidx = R0, wbase = R0;
  // block id of flat tile idx; tiles of a window lie a few pairs past pp
  auto load_phys = [&](int idx) -> int {
    if (idx >= R1) return 0;
    const TilePos t = locate_from(P, Hkv, pp, idx);
    return a.block_tables[(size_t)t.s * a.max_blocks + t.b];
  };
  int phys_cur = load_phys(wbase + lane);
  int phys_next = load_phys(wbase + 32 + lane);

  auto issue = [&](int stage) {
    int phys = __shfl_sync(kFull, phys_cur, pidx - wbase);
    if (lane == 0) {
      if (phys < 0 || (int64_t)phys >= a.num_blocks) {
        flag_error(PA_DEVERR_BLOCK_RANGE);
        phys = 0;
      }
      unsigned char* st = wbuf + stage * kStageBytes;
      const uint32_t bar = smem_addr(&bars[stage]);
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, 4 * kHalfBytes);
      const int y = (int)(((int64_t)phys * Hkv + pp.h) * kBlock);
      tma_load_2d(smem_addr(st), &tmk, 0, y, bar);
      tma_load_2d(smem_addr(st + kHalfBytes), &tmk, 64, y, bar);
      tma_load_2d(smem_addr(st + 2 * kHalfBytes), &tmv, 0, y, bar);
      tma_load_2d(smem_addr(st + 3 * kHalfBytes), &tmv, 64, y, bar);
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

  // ---- consumer --------------------------------------------------------------
  TilePos cp = locate(P, S, Hkv, R0);
  const int r0 = lane >> 2, r1 = r0 + 8;  // the two accumulator rows of this lane
  const int quad = lane & 3;
  uint32_t qa[8][4];
  float o[16][4];
  float m_r[2], l_r[2];
  int lim[2] = {0, 0}, lim_min = 0, lq = 0, ctx = 0;
  int piece_b0 = 0;
  bool piece_first = true;

  int k = 0;
  for (int idx = R0; idx < R1; ++idx, ++k) {
    const int stage = k % NSTAGE;
    const uint32_t parity = (uint32_t)(k / NSTAGE) & 1u;
    if (!mbar_wait_bounded(smem_addr(&bars[stage]), parity)) {
      for (int j = k + 1; j < k + NSTAGE && R0 + j < pidx; ++j)
        mbar_wait_bounded(smem_addr(&bars[j % NSTAGE]), (uint32_t)(j / NSTAGE) & 1u);
      return;
    }
    unsigned char* st = wbuf + stage * kStageBytes;
    const uint32_t sK = smem_addr(st), sV = smem_addr(st + 2 * kHalfBytes);
    const bool first = (idx == R0) || (cp.b == 0);
    if (first) {
      ctx = P.ctx[cp.s];
      lq = P.qstart[cp.s + 1] - P.qstart[cp.s];
      // Q fragments straight from global memory: row r of the tile is token
      // r / G, head r % G of this KV head. Rows past the sequence's last query
      // token are padding and stay zero (never written out).
      {
        const uint32_t* qrow[2] = {nullptr, nullptr};
        const int rws[2] = {r0, r1};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int tok = cp.qt * QT + rws[i] / G;
          if (tok < lq)
            qrow[i] = reinterpret_cast<const uint32_t*>(
                a.q + (((int64_t)P.qstart[cp.s] + tok) * Hq + (int64_t)cp.h * G + rws[i] % G) *
                          kHeadDim);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int c = kk * 8 + quad;  // 32-bit word of dims kk*16 + 2*quad
          qa[kk][0] = qrow[0] ? __ldg(qrow[0] + c) : 0u;
          qa[kk][1] = qrow[1] ? __ldg(qrow[1] + c) : 0u;
          qa[kk][2] = qrow[0] ? __ldg(qrow[0] + c + 4) : 0u;
          qa[kk][3] = qrow[1] ? __ldg(qrow[1] + c + 4) : 0u;
        }
      }
#pragma unroll
      for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
      m_r[0] = m_r[1] = neg_inf();
      l_r[0] = l_r[1] = 0.f;
      const int rows[2] = {r0, r1};
      // key limit of each row; padding rows (zero Q) need none
      int lv[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int tok = cp.qt * QT + rows[i] / G;
        const bool valid = tok < lq;
        lim[i] = valid ? (a.causal ? ctx - lq + tok + 1 : ctx) : 0x7fffffff;
        lv[i] = valid ? lim[i] : 0x7fffffff;
      }
      int mn = min(lv[0], lv[1]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) mn = min(mn, __shfl_xor_sync(kFull, mn, off));
      lim_min = mn;
      piece_b0 = cp.b;
      piece_first = (idx == R0);
    }
    const int key0 = cp.b * kBlock;
    // keys past the context may hold anything: zero those V rows so that
    // P = 0 never meets a NaN in the PV product
    if (key0 + kBlock > ctx) {
      const int zr = ctx - key0;  // first row to clear
      for (int i = lane; i < (kBlock - zr) * 16; i += 32) {
        const int row = zr + (i >> 4), c = i & 15;
        *reinterpret_cast<uint4*>(st + 2 * kHalfBytes + (c >> 3) * kHalfBytes + row * 128 +
                                  (c & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
      // compiler barrier: the (volatile) ldmatrix reads below stay after the stores
      asm volatile("" ::: "memory");
    }

    // ---- S = Q K^T (16 rows x 16 keys) -------------------------------------------
    float s[2][4];
    {
      // two independent accumulation chains per key group (even / odd k-steps)
      float sx[2][4];
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[n][e] = sx[n][e] = 0.f;
      const int mi = lane >> 3, rr = lane & 7;
      const int key = (mi >> 1) * 8 + rr;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int c = 2 * kk + (mi & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sK + (c >> 3) * kHalfBytes + swz(key, c & 7), b0, b1, b2, b3);
        if (kk & 1) {
          mma_bf16_16816(sx[0], qa[kk], b0, b1);
          mma_bf16_16816(sx[1], qa[kk], b2, b3);
        } else {
          mma_bf16_16816(s[0], qa[kk], b0, b1);
          mma_bf16_16816(s[1], qa[kk], b2, b3);
        }
      }
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[n][e] += sx[n][e];
    }
    // ---- mask, online softmax ----------------------------------------------------
    const bool need_mask = key0 + kBlock > lim_min;
#pragma unroll
    for (int n = 0; n < 2; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = s[n][e] * a.scale_log2;
        if (need_mask) {
          const int key = key0 + n * 8 + quad * 2 + (e & 1);
          if (key >= lim[e >> 1]) v = neg_inf();
        }
        s[n][e] = v;
      }
    }
    float alpha[2], mref[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float mx = fmaxf(fmaxf(s[0][2 * i], s[0][2 * i + 1]), fmaxf(s[1][2 * i], s[1][2 * i + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
      const float mn = fmaxf(m_r[i], mx);
      mref[i] = mn == neg_inf() ? 0.f : mn;
      alpha[i] = ex2(m_r[i] - mref[i]);
      m_r[i] = mn;
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int n = 0; n < 2; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = ex2(s[n][e] - mref[e >> 1]);
        s[n][e] = p;
        rs[e >> 1] += p;
      }
    }
    l_r[0] = l_r[0] * alpha[0] + rs[0];
    l_r[1] = l_r[1] * alpha[1] + rs[1];
    if (__any_sync(kFull, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        o[n][0] *= alpha[0];
        o[n][1] *= alpha[0];
        o[n][2] *= alpha[1];
        o[n][3] *= alpha[1];
      }
    }
    // ---- O += P V ----------------------------------------------------------------------
    uint32_t pa4[4];
    pa4[0] = cvt_bf16x2(s[0][0], s[0][1]);
    pa4[1] = cvt_bf16x2(s[0][2], s[0][3]);
    pa4[2] = cvt_bf16x2(s[1][0], s[1][1]);
    pa4[3] = cvt_bf16x2(s[1][2], s[1][3]);
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int key = (mi & 1) * 8 + rr;
#pragma unroll
      for (int cpair = 0; cpair < 8; ++cpair) {
        const int c = 2 * cpair + (mi >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_trans(sV + (c >> 3) * kHalfBytes + swz(key, c & 7), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * cpair], pa4, b0, b1);
        mma_bf16_16816(o[2 * cpair + 1], pa4, b2, b3);
      }
    }
    __syncwarp();

    if (pidx < R1) issue(stage);

    const bool last = (idx == R1 - 1) || (cp.b == cp.nt - 1);
    if (last) {
      float lt[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float x = l_r[i];
        x += __shfl_xor_sync(kFull, x, 1);
        x += __shfl_xor_sync(kFull, x, 2);
        lt[i] = x;
      }
      const bool complete = (piece_b0 == 0) && (cp.b == cp.nt - 1);
      const int rows[2] = {r0, r1};
      if (complete) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int tok = cp.qt * QT + rows[i] / G;
          if (tok >= lq) continue;
          const int g = rows[i] % G;
          const int64_t orow = ((int64_t)P.qstart[cp.s] + tok) * Hq + (int64_t)cp.h * G + g;
          const float inv = lt[i] > 0.f ? 1.f / lt[i] : 0.f;
          uint16_t* dst = a.out + orow * kHeadDim + quad * 2;
#pragma unroll
          for (int n = 0; n < 16; ++n)
            *reinterpret_cast<uint32_t*>(dst + n * 8) =
                cvt_bf16x2(o[n][2 * i] * inv, o[n][2 * i + 1] * inv);
          if (a.lse && quad == 0)
            a.lse[orow] = lt[i] > 0.f ? (m_r[i] + lg2(lt[i])) * kLn2 : neg_inf();
        }
      } else {
        const size_t slot = (size_t)w * 2 + (piece_first ? 0 : 1);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float inv = lt[i] > 0.f ? 1.f / lt[i] : 0.f;
          float* dst = a.part_o + (slot * kRows + rows[i]) * kHeadDim + quad * 2;
#pragma unroll
          for (int n = 0; n < 16; ++n)
            *reinterpret_cast<float2*>(dst + n * 8) =
                make_float2(o[n][2 * i] * inv, o[n][2 * i + 1] * inv);
          if (quad == 0)
            a.part_lse[slot * kRows + rows[i]] =
                lt[i] > 0.f ? (m_r[i] + lg2(lt[i])) * kLn2 : neg_inf();
        }
      }
    }
    if (idx + 1 < R1) advance(P, S, Hkv, cp);
  }
}

template <int NWARPS, int NSTAGE>
__global__ void __launch_bounds__(NWARPS * 32)
    paged_varlen_kernel(const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const VarlenArgs a) {
  varlen_body<NWARPS, NSTAGE>(tmk, tmv, a);
  // late: thread 0 of each CTA waits for the grid ahead on the way out, so
  // this grid never completes before it
  if (a.late && threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Merge the pieces of (sequence, query tile, KV head) segments cut by the
// balanced ranges. One CTA per worker boundary; a warp merges four rows at
// once (eight lanes per row, sixteen dims per lane), online over the pieces,
// four pieces at a time with all their loads in flight. Partials are read
// through L2 (ld.global.cg): other SMs wrote them.
constexpr int kFixWarps = kRows / 4;

__global__ void __launch_bounds__(kFixWarps * 32)
    varlen_fixup_kernel(const int* __restrict__ desc, const float* __restrict__ part_o,
                        const float* __restrict__ part_lse,
                        const int32_t* __restrict__ cu_seqlens_q, int num_workers, int Hq, int G,
                        int QT, uint16_t* __restrict__ out, float* __restrict__ lse) {
  // the next grid in the stream may start its own preparation now; it waits
  // for this grid before it reads anything this grid writes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int w = blockIdx.x;
  if (w >= num_workers) return;
  const int* d = desc + (size_t)w * kDescInts;
  const int s = __ldcg(d);
  if (s < 0) return;
  const int qt = __ldcg(d + 1), h = __ldcg(d + 2), last = __ldcg(d + 3),
            slot_prev = __ldcg(d + 4);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = warp * 4 + (lane >> 3);
  const int d0 = (lane & 7) * 16;
  const int q0 = cu_seqlens_q[s], lq = cu_seqlens_q[s + 1] - q0;
  const int tok = qt * QT + r / G;
  if (tok >= lq) return;
  const int npieces = last - w + 2;  // workers w-1 .. last
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
        const size_t sl = (size_t)(w - 1 + i0 + u) * 2 + (i0 + u == 0 ? slot_prev : 0);
        li[u] = __ldcg(part_lse + sl * kRows + r);
        const float4* src = reinterpret_cast<const float4*>(part_o + (sl * kRows + r) * kHeadDim + d0);
#pragma unroll
        for (int k = 0; k < 4; ++k) x[u][k] = __ldcg(src + k);
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
  const float LSE = sum > 0.f ? m + lg2(sum) * kLn2 : neg_inf();
  const int64_t orow = ((int64_t)q0 + tok) * Hq + (int64_t)h * G + r % G;
  uint4* dst = reinterpret_cast<uint4*>(out + orow * kHeadDim + d0);
  dst[0] = make_uint4(cvt_bf16x2(acc[0] * inv, acc[1] * inv), cvt_bf16x2(acc[2] * inv, acc[3] * inv),
                      cvt_bf16x2(acc[4] * inv, acc[5] * inv), cvt_bf16x2(acc[6] * inv, acc[7] * inv));
  dst[1] = make_uint4(cvt_bf16x2(acc[8] * inv, acc[9] * inv), cvt_bf16x2(acc[10] * inv, acc[11] * inv),
                      cvt_bf16x2(acc[12] * inv, acc[13] * inv), cvt_bf16x2(acc[14] * inv, acc[15] * inv));
  if (lse && (lane & 7) == 0) lse[orow] = LSE;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
constexpr int kWarps = 6;
constexpr int kStages = 3;  // one CTA per SM: 6 warps x 3 stages of 8 KB (best of a warps x stages sweep)

struct VarlenGeometry {
  int grid = 0, workers = 0, npairs_cap = 0;
  size_t smem = 0, ws_desc = 0, ws_lse = 0, ws_o = 0, ws_bytes = 0;
};

int varlen_geometry(const pa_shape* sh, int64_t num_q_tokens, int max_q_len,
                    VarlenGeometry* g) {
  DeviceInfo dev;
  if (!current_device_info(&dev)) return PA_ERR_CUDA;
  const int S = sh->num_seqs;
  const int G = sh->num_q_heads / sh->num_kv_heads, QT = kRows / G;
  const int64_t cap1 = (int64_t)S * ((max_q_len + QT - 1) / QT);
  const int64_t cap2 = (num_q_tokens + QT - 1) / QT + S;
  const int64_t cap = cap1 < cap2 ? cap1 : cap2;
  if (cap > (1 << 22)) return PA_ERR_UNSUPPORTED;
  g->npairs_cap = (int)(cap < 1 ? 1 : cap);
  const size_t plan = sizeof(int) * ((size_t)g->npairs_cap + 1 + 3 * (size_t)S + 2 + 40);
  g->smem = 1024 + (size_t)kWarps * kStages * kStageBytes + (size_t)kWarps * kStages * 8 + plan;
  if (g->smem > (size_t)dev.max_smem_optin) return PA_ERR_UNSUPPORTED;
  const void* kern = reinterpret_cast<const void*>(paged_varlen_kernel<kWarps, kStages>);
  int per_sm = 0;
  if (!kernel_occupancy(kern, kWarps * 32, g->smem, &per_sm) || per_sm <= 0) return PA_ERR_CUDA;
  g->grid = dev.num_sms * per_sm;
  g->workers = g->grid * kWarps;
  g->ws_desc = round_up(sizeof(int) * kDescInts * (size_t)g->workers, 256);
  g->ws_lse = round_up(sizeof(float) * 2 * kRows * (size_t)g->workers, 256);
  g->ws_o = round_up(sizeof(float) * 2 * kRows * kHeadDim * (size_t)g->workers, 256);
  g->ws_bytes = g->ws_desc + g->ws_lse + g->ws_o;
  return PA_OK;
}

int check_varlen_args(const pa_shape* shape, int64_t num_q_tokens, int max_q_len) {
  int rc = check_shape_common(shape);
  if (rc != PA_OK) return rc;
  const int G = shape->num_q_heads / shape->num_kv_heads;
  if (G > kRows || kRows % G != 0) return PA_ERR_UNSUPPORTED;
  if (num_q_tokens < 0 || max_q_len < 0) return PA_ERR_ARG;
  if (num_q_tokens > 0x3fffffff) return PA_ERR_ARG;
  if (shape->num_blocks * shape->num_kv_heads * kBlock > 0x7fffffff) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_pool_map(CUtensorMap* map, const void* pool, int64_t rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kBlock};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

unsigned take_error_word_varlen(cudaStream_t stream, int* rc) {
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

extern "C" size_t pa_decode_varlen_workspace_size(const pa_shape* shape, int64_t num_q_tokens,
                                                  int max_q_len) {
  if (check_varlen_args(shape, num_q_tokens, max_q_len) != PA_OK) return 0;
  if (shape->num_seqs == 0 || num_q_tokens == 0) return 0;
  VarlenGeometry g;
  if (varlen_geometry(shape, num_q_tokens, max_q_len, &g) != PA_OK) return 0;
  PrefillTcGeometry tg;
  if (prefill_tc_geometry(shape, num_q_tokens, max_q_len, &tg) != PA_OK) return 0;
  return g.ws_bytes + tg.ws_bytes;
}

extern "C" int pa_decode_varlen(const pa_bf16* q, const pa_bf16* k_cache, const pa_bf16* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens,
                                const int32_t* cu_seqlens_q, int64_t num_q_tokens,
                                int max_q_len, int causal, float scale, pa_bf16* out, float* lse,
                                const pa_shape* shape, void* workspace, size_t workspace_bytes,
                                void* stream) {
  pa::NvtxRange nvtx_range("pa_decode_varlen");
  int rc = check_varlen_args(shape, num_q_tokens, max_q_len);
  if (rc != PA_OK) return rc;
  if (shape->num_seqs == 0 || num_q_tokens == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !cu_seqlens_q || !out)
    return PA_ERR_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(cu_seqlens_q, 4) ||
      (lse && !aligned(lse, 4)))
    return PA_ERR_ARG;
  if (!(scale == scale)) return PA_ERR_ARG;
  VarlenGeometry g;
  rc = varlen_geometry(shape, num_q_tokens, max_q_len, &g);
  if (rc != PA_OK) return rc;
  PrefillTcGeometry tg;
  rc = prefill_tc_geometry(shape, num_q_tokens, max_q_len, &tg);
  if (rc != PA_OK) return rc;
  if (!workspace || workspace_bytes < g.ws_bytes + tg.ws_bytes || !aligned(workspace, 256))
    return PA_ERR_WORKSPACE;
  const int64_t rows = shape->num_blocks * shape->num_kv_heads * kBlock;
  CUtensorMap tmk, tmv;
  if (!make_pool_map(&tmk, k_cache, rows) || !make_pool_map(&tmv, v_cache, rows))
    return PA_ERR_CUDA;

  VarlenArgs a;
  a.q = q;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.cu_seqlens_q = cu_seqlens_q;
  a.out = out;
  a.lse = lse;
  a.scale_log2 = (float)((double)scale * 1.4426950408889634);
  a.S = shape->num_seqs;
  a.Hq = shape->num_q_heads;
  a.Hkv = shape->num_kv_heads;
  a.G = a.Hq / a.Hkv;
  a.QT = kRows / a.G;
  a.max_blocks = shape->max_blocks_per_seq;
  a.num_blocks = shape->num_blocks;
  a.num_q_tokens = num_q_tokens;
  a.causal = causal ? 1 : 0;
  a.npairs_cap = g.npairs_cap;
  a.num_workers = g.workers;
  a.max_lq = tg.enabled ? kTcMinQLen - 1 : 0x7fffffff;
  char* ws = static_cast<char*>(workspace);
  a.desc = reinterpret_cast<int*>(ws);
  a.part_lse = reinterpret_cast<float*>(ws + g.ws_desc);
  a.part_o = reinterpret_cast<float*>(ws + g.ws_desc + g.ws_lse);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Sequences with long query chunks (prefill) run as tcgen05 tiles of 128
  // rows, the others (verify) on the mma.sync kernel; the prefill grid goes
  // first. When the batch surely holds short sequences (fewer than
  // kTcMinQLen query tokens per sequence on average), the two grids run side
  // by side: the prefill grid keeps the K of its CTAs that overlap_split
  // gives (one per SM; the rest leave at once), the verify grid follows it as
  // a late dependent and deals its work to the CTAs that land on the other
  // SMs, and the prefill merge moves behind the verify grid.
  // Otherwise (prefill-only batches) the prefill merge follows its own grid
  // directly, one grid-completion hop earlier.
  const bool overlap = tg.enabled && num_q_tokens < (int64_t)kTcMinQLen * shape->num_seqs;
  a.late = overlap ? 1 : 0;
  a.split = overlap ? tg.grid : 0;
  if (tg.enabled) {
    rc = launch_prefill_tc(tg, q, k_cache, v_cache, block_tables, context_lens, cu_seqlens_q,
                           num_q_tokens, causal, scale, out, lse, shape, ws + g.ws_bytes, st,
                           kTcMinQLen, nullptr, nullptr, /*parts=*/overlap ? 1 : 3,
                           /*split=*/overlap ? 1 : 0);
    if (rc != PA_OK) return rc;
  }
  if (launch_dependent(paged_varlen_kernel<kWarps, kStages>, dim3(g.grid), dim3(kWarps * 32),
                       g.smem, st, tmk, tmv, a) != cudaSuccess)
    return PA_ERR_CUDA;
  if (overlap) {
    rc = launch_prefill_tc(tg, q, k_cache, v_cache, block_tables, context_lens, cu_seqlens_q,
                           num_q_tokens, causal, scale, out, lse, shape, ws + g.ws_bytes, st,
                           kTcMinQLen, nullptr, nullptr, /*parts=*/2, /*split=*/1);
    if (rc != PA_OK) return rc;
  }
  if (launch_dependent(varlen_fixup_kernel, dim3(g.workers), dim3(kFixWarps * 32), 0, st,
                       (const int*)a.desc, (const float*)a.part_o, (const float*)a.part_lse,
                       cu_seqlens_q, g.workers, a.Hq, a.G, a.QT, (uint16_t*)out,
                       lse) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}
