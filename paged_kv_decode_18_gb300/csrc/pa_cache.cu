// pa_cache.cu -- slot-mapped write of the step's new K/V rows into the paged
// pool (LLM inference engine work-log, "KV Cache > The Idea": the new K and V
// are appended to the cache before the new queries attend; course README
// "Build an LLM Inference Engine From Scratch": chunked prefill gives a
// bit-identical cache).
//
// bf16 pool: a byte copy -- each thread moves one 16-byte chunk of K and the
// matching chunk of V. Reads of k/v are fully coalesced; each (token, KV
// head) row lands as one contiguous 256-byte run of the (block, KV head)
// tile. 8-bit pools (int8, FP8 E4M3; course README, curriculum rows "The
// Machine" and "Memory & KV Cache": fp8, quantization): one warp quantises
// one row with its own fp32 scale and writes 128 code bytes plus the scale
// into the tile.
#include "pa_device.cuh"
#include "pa_host.h"

namespace pa {
namespace {

constexpr int kChunksPerRow = kHeadDim * 2 / 16;  // 16-byte chunks per (token, head) row

__global__ void reshape_and_cache_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                         const int64_t* __restrict__ slots, int64_t total_chunks,
                                         int Hkv, int64_t num_slots, uint4* __restrict__ k_cache,
                                         uint4* __restrict__ v_cache) {
  // launched as a programmatic dependent: wait for the previous grid (which may
  // produce k, v or the slots), then let a dependent grid queued behind this
  // one (decode in pa_append_decode) start its own preparation; that grid
  // reads only call inputs before it waits for this one
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total_chunks) return;
  const int per_token = Hkv * kChunksPerRow;
  const int64_t t = i / per_token;
  const int r = (int)(i - t * per_token);
  const int h = r / kChunksPerRow, c = r % kChunksPerRow;
  const int64_t slot = slots[t];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (r == 0) flag_error(PA_DEVERR_SLOT_RANGE);
    return;
  }
  const int64_t blk = slot / kBlock, off = slot % kBlock;
  const int64_t dst = (((blk * Hkv + h) * kBlock + off) * kChunksPerRow) + c;
  k_cache[dst] = k[i];
  v_cache[dst] = v[i];
}

// Quantising write (INT8 KV): one warp per (token, KV head) row of 128 values.
// Symmetric, one fp32 scale per row: amax = max |x|, q = rint(x * (127 / amax))
// clamped to [-127, 127], scale = amax / 127; a zero row stores q = 0 and
// scale = 0. Division and product are IEEE-rounded fp32 operations (explicit
// _rn intrinsics, no contraction), rint rounds half to even. The row lands
// as 128 contiguous bytes of the (block, KV head) int8 tile and one float of
// the same tile's scale slots.
__device__ __forceinline__ void quantize_row_to(const uint2 x, int lane, int8_t* __restrict__ dst,
                                                float* __restrict__ scale_dst) {
  const float f0 = bf_lo(x.x), f1 = bf_hi(x.x), f2 = bf_lo(x.y), f3 = bf_hi(x.y);
  float amax = fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
  uint32_t packed = 0u;
  if (amax > 0.f) {
    const float inv = __fdiv_rn(127.f, amax);
    const float fs[4] = {f0, f1, f2, f3};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float t = fminf(fmaxf(rintf(__fmul_rn(fs[j], inv)), -127.f), 127.f);
      packed |= ((uint32_t)(int)t & 0xffu) << (8 * j);
    }
  }
  reinterpret_cast<uint32_t*>(dst)[lane] = packed;
  if (lane == 0) *scale_dst = amax > 0.f ? __fdiv_rn(amax, 127.f) : 0.f;
}

// Quantising write (FP8 E4M3 KV): as the int8 write, with the row's amax
// mapped to the largest finite E4M3 value 448: y = x * (448 / amax) in IEEE
// fp32, code = the nearest E4M3 value of y (ties to the even code), saturated
// to +-448 (the hardware conversion with .satfinite), scale = amax / 448. A
// zero row stores code 0 and scale 0. The codes never hold the NaN patterns.
__device__ __forceinline__ uint32_t e4m3x2_of(float lo, float hi) {
  uint16_t c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(hi), "f"(lo));
  return c;
}

__device__ __forceinline__ void quantize_row_f8_to(const uint2 x, int lane,
                                                   uint8_t* __restrict__ dst,
                                                   float* __restrict__ scale_dst) {
  const float f0 = bf_lo(x.x), f1 = bf_hi(x.x), f2 = bf_lo(x.y), f3 = bf_hi(x.y);
  float amax = fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
  uint32_t packed = 0u;
  if (amax > 0.f) {
    const float inv = __fdiv_rn(448.f, amax);
    packed = e4m3x2_of(__fmul_rn(f0, inv), __fmul_rn(f1, inv)) |
             (e4m3x2_of(__fmul_rn(f2, inv), __fmul_rn(f3, inv)) << 16);
  }
  reinterpret_cast<uint32_t*>(dst)[lane] = packed;
  if (lane == 0) *scale_dst = amax > 0.f ? __fdiv_rn(amax, 448.f) : 0.f;
}

// One warp per (token, KV head) row; FP8 selects the E4M3 codes, else int8.
template <bool FP8>
__global__ void reshape_and_cache_q8_kernel(const uint2* __restrict__ k,
                                            const uint2* __restrict__ v,
                                            const int64_t* __restrict__ slots, int64_t rows,
                                            int Hkv, int64_t num_slots,
                                            uint8_t* __restrict__ k_cache,
                                            uint8_t* __restrict__ v_cache) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;  // warp-uniform
  const int64_t t = row / Hkv;
  const int h = (int)(row - t * Hkv);
  const int64_t slot = slots[t];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (lane == 0) flag_error(PA_DEVERR_SLOT_RANGE);
    return;
  }
  const int64_t blk = slot / kBlock, off = slot % kBlock;
  // tile (blk, h): 16 rows of 128 codes, then the 16 rows' fp32 scales
  const int64_t tile = (blk * Hkv + h) * kInt8TileBytes;
  // lane reads dims 4*lane .. 4*lane+3 (8 bytes): the warp reads the 256-byte row
  const uint2 xk = k[row * 32 + lane], xv = v[row * 32 + lane];
  float* k_scale = reinterpret_cast<float*>(k_cache + tile + kBlock * kHeadDim) + off;
  float* v_scale = reinterpret_cast<float*>(v_cache + tile + kBlock * kHeadDim) + off;
  if constexpr (FP8) {
    quantize_row_f8_to(xk, lane, k_cache + tile + off * kHeadDim, k_scale);
    quantize_row_f8_to(xv, lane, v_cache + tile + off * kHeadDim, v_scale);
  } else {
    quantize_row_to(xk, lane, reinterpret_cast<int8_t*>(k_cache + tile) + off * kHeadDim,
                    k_scale);
    quantize_row_to(xv, lane, reinterpret_cast<int8_t*>(v_cache + tile) + off * kHeadDim,
                    v_scale);
  }
}

template <bool FP8>
int launch_cache_write_q8(const pa_bf16* k, const pa_bf16* v, const int64_t* slot_mapping,
                          int64_t num_tokens, uint8_t* k_cache, uint8_t* v_cache,
                          const pa_shape* shape, cudaStream_t st) {
  int rc = check_shape_common(shape);
  if (rc != PA_OK) return rc;
  if (num_tokens < 0) return PA_ERR_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PA_ERR_ARG;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8))
    return PA_ERR_ARG;
  const int64_t rows = num_tokens * shape->num_kv_heads;
  const int wpb = 8;
  const int64_t blocks = (rows + wpb - 1) / wpb;
  if (blocks > 0x7fffffff) return PA_ERR_ARG;
  if (launch_dependent(reshape_and_cache_q8_kernel<FP8>, dim3((unsigned)blocks), dim3(wpb * 32),
                       0, st, reinterpret_cast<const uint2*>(k),
                       reinterpret_cast<const uint2*>(v), slot_mapping, rows,
                       shape->num_kv_heads, shape->num_blocks * shape->block_size, k_cache,
                       v_cache) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

}  // namespace

int launch_cache_write(const pa_bf16* k, const pa_bf16* v, const int64_t* slot_mapping,
                       int64_t num_tokens, pa_bf16* k_cache, pa_bf16* v_cache,
                       const pa_shape* shape, cudaStream_t st) {
  int rc = check_shape_common(shape);
  if (rc != PA_OK) return rc;
  if (num_tokens < 0) return PA_ERR_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PA_ERR_ARG;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8))
    return PA_ERR_ARG;
  const int64_t total = num_tokens * shape->num_kv_heads * kChunksPerRow;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 0x7fffffff) return PA_ERR_ARG;
  if (launch_dependent(reshape_and_cache_kernel, dim3((unsigned)blocks), dim3(threads), 0, st,
                       reinterpret_cast<const uint4*>(k), reinterpret_cast<const uint4*>(v),
                       slot_mapping, total, shape->num_kv_heads,
                       shape->num_blocks * shape->block_size, reinterpret_cast<uint4*>(k_cache),
                       reinterpret_cast<uint4*>(v_cache)) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

unsigned take_error_word_cache(cudaStream_t stream, int* rc) {
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

extern "C" int pa_reshape_and_cache(const pa_bf16* k, const pa_bf16* v,
                                    const int64_t* slot_mapping, int64_t num_tokens,
                                    pa_bf16* k_cache, pa_bf16* v_cache, const pa_shape* shape,
                                    void* stream) {
  pa::NvtxRange nvtx_range("pa_reshape_and_cache");
  return launch_cache_write(k, v, slot_mapping, num_tokens, k_cache, v_cache, shape,
                            static_cast<cudaStream_t>(stream));
}

extern "C" int pa_reshape_and_cache_int8(const pa_bf16* k, const pa_bf16* v,
                                         const int64_t* slot_mapping, int64_t num_tokens,
                                         uint8_t* k_cache, uint8_t* v_cache,
                                         const pa_shape* shape, void* stream) {
  pa::NvtxRange nvtx_range("pa_reshape_and_cache_int8");
  return launch_cache_write_q8<false>(k, v, slot_mapping, num_tokens, k_cache, v_cache, shape,
                                      static_cast<cudaStream_t>(stream));
}

extern "C" int pa_reshape_and_cache_fp8(const pa_bf16* k, const pa_bf16* v,
                                        const int64_t* slot_mapping, int64_t num_tokens,
                                        uint8_t* k_cache, uint8_t* v_cache,
                                        const pa_shape* shape, void* stream) {
  pa::NvtxRange nvtx_range("pa_reshape_and_cache_fp8");
  return launch_cache_write_q8<true>(k, v, slot_mapping, num_tokens, k_cache, v_cache, shape,
                                     static_cast<cudaStream_t>(stream));
}
