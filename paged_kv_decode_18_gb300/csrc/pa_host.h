// pa_host.h -- host-side helpers shared by the translation units of
// libpagedattn: status plumbing, shape checks, cached device properties.
#pragma once

#include <cuda.h>
#include <nvtx3/nvToolsExt.h>

#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <utility>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  int max_smem_optin = 0;  // bytes of dynamic shared memory a CTA may opt in to
};

// Properties of the current device (queried once per device, then cached).
// Returns false if a CUDA call fails.
inline bool current_device_info(DeviceInfo* out) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev].device != dev) {
    DeviceInfo d;
    d.device = dev;
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return false;
    if (cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
        cudaSuccess)
      return false;
    cache[dev] = d;
  }
  *out = cache[dev];
  return true;
}

// A kernel's dynamic shared-memory limit is raised to the device maximum once
// per (kernel, device); the launches pass their actual size.
inline bool raise_smem_limit(const void* fn) {
  DeviceInfo dev;
  if (!current_device_info(&dev)) return false;
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({fn, dev.device})) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           dev.max_smem_optin) != cudaSuccess)
    return false;
  done.insert({fn, dev.device});
  return true;
}

// Resident CTAs per SM of a kernel for a block size and dynamic shared-memory
// size, queried once per (kernel, device, threads, bytes) and then cached:
// the host path of a call stays free of driver queries.
inline bool kernel_occupancy(const void* fn, int threads, size_t smem, int* per_sm) {
  if (!raise_smem_limit(fn)) return false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, int, size_t>, int> cache;
  const auto key = std::make_tuple(fn, dev, threads, smem);
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) {
      *per_sm = it->second;
      return true;
    }
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess)
    return false;
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = n;
  *per_sm = n;
  return true;
}

inline bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Checks of the shape fields every call uses.
inline int check_shape_common(const pa_shape* s) {
  if (!s) return PA_ERR_ARG;
  if (s->num_seqs < 0 || s->num_q_heads <= 0 || s->num_kv_heads <= 0 || s->head_dim <= 0 ||
      s->block_size <= 0 || s->max_blocks_per_seq < 0 || s->num_blocks < 0)
    return PA_ERR_ARG;
  if (s->num_q_heads % s->num_kv_heads != 0) return PA_ERR_ARG;
  if (s->head_dim != 128 || s->block_size != 16) return PA_ERR_UNSUPPORTED;
  // flat tile indices and slot numbers are kept in 32-bit ints
  if (static_cast<int64_t>(s->max_blocks_per_seq) * s->block_size > (1 << 30)) return PA_ERR_ARG;
  if (s->num_blocks * s->num_kv_heads * s->block_size >= (int64_t(1) << 40)) return PA_ERR_ARG;
  return PA_OK;
}

// A named NVTX range around a C-ABI call (visible in Nsight timelines; a
// no-op when no tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Launch a kernel as a programmatic dependent of the previous grid on the
// stream (it may start before that grid ends and waits inside).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// fp32 row output of an attention launch, as one slot of a split-K partial
// layout: row r (= token * Hq + head) goes to o[(r * stride + slot) * D] and
// lse[r * stride + slot] (normalised o, natural-log lse).
struct RowsOut {
  float* o = nullptr;
  float* lse = nullptr;
  int stride = 1;
  int slot = 0;
  int64_t tokens = 0;  // output tokens (rows / Hq); a mapped token outside is skipped
};

// Slot-mapped cache write (pa_cache.cu), as pa_reshape_and_cache.
int launch_cache_write(const pa_bf16* k, const pa_bf16* v, const int64_t* slot_mapping,
                       int64_t num_tokens, pa_bf16* k_cache, pa_bf16* v_cache,
                       const pa_shape* shape, cudaStream_t st);

// Balanced decode (pa_decode with num_splits 0) writing fp32 rows (pa_decode.cu).
// late: see DecodeArgs::late; max_sms > 0 sizes the grid for that many SMs.
int decode_rows(const pa_bf16* q, const pa_bf16* k_cache, const pa_bf16* v_cache,
                const int32_t* block_tables, const int32_t* context_lens, float scale,
                const pa_shape* shape, const RowsOut& rows, void* workspace,
                size_t workspace_bytes, cudaStream_t st, int late = 0, int max_sms = 0);
size_t decode_rows_workspace_size(const pa_shape* shape, int max_sms);

// ---------------------------------------------------------------------------
// tensor maps (pa_varlen.cu)
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
// 2-D view of one pool array: [num_blocks * Hkv * 16 rows][128] bf16, boxes of
// 16 rows x 64 dims, 128-byte swizzle.
bool make_pool_map(CUtensorMap* map, const void* pool, int64_t rows);

// ---------------------------------------------------------------------------
// tcgen05 prefill path (pa_prefill_tc.cu): sequences with q_len >= this go
// there; the mma.sync varlen kernel takes the shorter ones (verify).
// ---------------------------------------------------------------------------
constexpr int kTcMinQLen = 32;

struct PrefillTcGeometry {
  bool enabled = false;
  int grid = 0, workers = 0, npairs_cap = 0, QTb = 0;
  size_t smem = 0, fixup_smem = 0, ws_lse = 0, ws_o = 0, ws_bytes = 0;
};

// min_q_len: sequences with a shorter query window are left to another kernel.
// max_ctas > 0 caps the grid (one CTA per SM) at that many CTAs.
int prefill_tc_geometry(const pa_shape* sh, int64_t num_q_tokens, int max_q_len,
                        PrefillTcGeometry* g, int min_q_len = kTcMinQLen, int max_ctas = 0);
// rows / row_map (optional): write fp32 rows instead of out / lse, query
// token i of q landing as token row_map[i] (row_map may be null: identity).
int launch_prefill_tc(const PrefillTcGeometry& g, const pa_bf16* q, const pa_bf16* k_cache,
                      const pa_bf16* v_cache, const int32_t* block_tables,
                      const int32_t* context_lens, const int32_t* cu_seqlens_q,
                      int64_t num_q_tokens, int causal, float scale, pa_bf16* out, float* lse,
                      const pa_shape* sh, void* workspace, cudaStream_t st,
                      int min_q_len = kTcMinQLen, const RowsOut* rows = nullptr,
                      const int32_t* row_map = nullptr, int parts = 3, int split = 0);
// parts: bit 0 launches the attention grid, bit 1 its merge grid.

// Each TU that owns kernels exposes the reader of its device error word.
unsigned take_error_word_cache(cudaStream_t stream, int* rc);
unsigned take_error_word_decode(cudaStream_t stream, int* rc);
unsigned take_error_word_varlen(cudaStream_t stream, int* rc);
unsigned take_error_word_prefill(cudaStream_t stream, int* rc);
unsigned take_error_word_cascade(cudaStream_t stream, int* rc);

}  // namespace pa
