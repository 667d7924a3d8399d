// pa_cascade.cu -- prefix-aware (cascade) decode: sequences that share the
// physical blocks of a prompt prefix attend that prefix once per group.
//
// Pages: course README "Build an LLM Inference Engine From Scratch",
// "What to build in what order" (prefix caching: the largest win per line
// of code when traffic shares prefixes) and "S20 - The Complete Engine",
// section "The conflicts" (prefix cache: reference-counted blocks shared by
// requests); the split-K claim "online softmax is exact; paged and split-K
// variants agree" makes the two halves mergeable.
//
// For a sequence s in group g (prefix of P_g tokens, a multiple of the block
// size, held in the same physical blocks by every member), attention over
// its context splits at P_g into two disjoint key ranges:
//   prefix: keys 0 .. P_g-1, shared by every member of g. Its K/V are read
//           once for the whole group: the members' query rows form one
//           non-causal multi-query problem (M = members x G rows per KV
//           head), run on the tcgen05 prefill tile;
//   suffix: keys P_g .. c_s-1, private. The balanced decode kernel runs on a
//           suffix view of the block table (row shifted by P_g / BS blocks,
//           context c_s - P_g).
// Each half writes (o, lse) as one fp32 split-K partial; the split-K merge
// combines them (an empty half has lse = -inf and weight 0). A sequence in
// no group has an empty prefix half and its whole context in the suffix.
#include "pa_device.cuh"
#include "pa_host.h"

namespace pa {
namespace {

struct CascadeLayout {
  size_t q_g = 0, prefix_bt = 0, suffix_bt = 0, suffix_cl = 0, part_o = 0, part_lse = 0,
         tc_ws = 0, dec_ws = 0, total = 0;
  PrefillTcGeometry tg;
  pa_shape tc_shape{}, suffix_shape{};
  size_t dec_ws_bytes = 0;
  int tc_ctas = 0;      // SMs given to the prefix half
  int suffix_sms = 0;   // SMs the suffix half's grid is sized for (0: all)
};

int cascade_layout(const pa_shape* sh, int num_groups, int num_members, int max_group_size,
                   int max_prefix_len, CascadeLayout* L) {
  const int S = sh->num_seqs, Hq = sh->num_q_heads;
  if (num_groups < 0 || num_members < 0 || max_group_size < 0 || max_prefix_len < 0)
    return PA_ERR_ARG;
  if (max_prefix_len % kBlock != 0) return PA_ERR_ARG;
  const int max_prefix_blocks = max_prefix_len / kBlock;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += round_up(bytes, 256);
    return at;
  };
  L->q_g = take((size_t)num_members * Hq * kHeadDim * 2);
  L->prefix_bt = take((size_t)num_groups * max_prefix_blocks * 4);
  L->suffix_bt = take((size_t)S * sh->max_blocks_per_seq * 4);
  L->suffix_cl = take((size_t)S * 4);
  L->part_o = take((size_t)S * Hq * 2 * kHeadDim * 4);
  L->part_lse = take((size_t)S * Hq * 2 * 4);
  // prefix half: the groups are the "sequences", members their query tokens
  L->tc_shape = *sh;
  L->tc_shape.num_seqs = num_groups;
  L->tc_shape.max_blocks_per_seq = max_prefix_blocks;
  if (num_groups > 0 && num_members > 0 && max_prefix_blocks > 0) {
    // The two halves run side by side: the prefix half on tc_ctas SMs (about
    // 12 of its 128 x 128 tiles per CTA, from an upper bound of its tile
    // count: the best of a sweep of 4..24 on a shared-prompt batch), the
    // suffix half on the others.
    DeviceInfo dev;
    if (!current_device_info(&dev)) return PA_ERR_CUDA;
    const int G = sh->num_q_heads / sh->num_kv_heads;
    const int qtb = 128 / (G > 0 ? G : 1);
    const int64_t qtiles = (num_members + qtb - 1) / qtb + num_groups;
    const int64_t tiles = qtiles * sh->num_kv_heads * ((max_prefix_len + 127) / 128);
    int64_t want = (tiles + 11) / 12;
    const int64_t cap = dev.num_sms / 2;
    L->tc_ctas = (int)(want < 8 ? 8 : (want > cap ? cap : want));
    L->suffix_sms = dev.num_sms - L->tc_ctas;
    const int rc = prefill_tc_geometry(&L->tc_shape, num_members, max_group_size, &L->tg, 1,
                                       L->tc_ctas);
    if (rc != PA_OK) return rc;
    if (!L->tg.enabled) return PA_ERR_UNSUPPORTED;
  } else {
    L->tg.enabled = false;
  }
  L->tc_ws = take(L->tg.enabled ? L->tg.ws_bytes : 0);
  L->suffix_shape = *sh;
  L->dec_ws_bytes = S > 0 ? decode_rows_workspace_size(sh, L->suffix_sms) : 0;
  if (S > 0 && L->dec_ws_bytes == 0) return PA_ERR_ARG;
  L->dec_ws = take(L->dec_ws_bytes);
  // the plain balanced decode over the whole contexts uses the workspace
  // from its start (policy PA_CASCADE_PLAIN, or PA_CASCADE_AUTO choosing it)
  const size_t plain = S > 0 ? decode_rows_workspace_size(sh, 0) : 0;
  L->total = off > plain ? off : plain;
  return PA_OK;
}

// Bytes of K/V rows the cascade saves at most: every member but the first of
// a group skips reading the group's prefix, at most max_prefix_len tokens.
// Measured on GB300 (shared-prompt batches of 16..128 sequences behind
// prefixes of 256..4096 tokens, against pa_decode): the cascade is faster
// once it saves about 256 MB per 64 members (its prefix tile and merge grow
// with the members); below that its extra phases cost more than the prefix
// reads they save, which plain decode mostly finds in L2.
constexpr int64_t kCascadeMinSavedBytes = int64_t(256) << 20;

bool cascade_pays(const pa_shape* sh, int num_groups, int num_members, int max_prefix_len) {
  const int64_t per_token = (int64_t)sh->num_kv_heads * sh->head_dim * 2 * 2;
  const int64_t saved = (int64_t)(num_members - num_groups) * max_prefix_len * per_token;
  const int64_t scale = num_members > 64 ? num_members : 64;
  return saved > 0 && saved * 64 >= kCascadeMinSavedBytes * scale;
}

// Everything the two halves need, in one grid-stride pass:
//   suffix block tables (row s shifted by its prefix blocks) and contexts;
//   the gathered query rows of the members, group by group;
//   each group's prefix block table (from its first member's row);
//   the (0, -inf) prefix partial of every sequence in no group;
// with the consistency checks of the group description.
__global__ void cascade_prep_kernel(const uint4* __restrict__ q, const int32_t* __restrict__ block_tables,
                                    const int32_t* __restrict__ context_lens,
                                    const int32_t* __restrict__ seq_group,
                                    const int32_t* __restrict__ cu_group,
                                    const int32_t* __restrict__ group_members,
                                    const int32_t* __restrict__ prefix_lens, int S, int Hq,
                                    int max_blocks, int num_groups, int num_members,
                                    int max_prefix_blocks, uint4* __restrict__ q_g,
                                    int32_t* __restrict__ prefix_bt,
                                    int32_t* __restrict__ suffix_bt,
                                    int32_t* __restrict__ suffix_cl, float* __restrict__ part_o,
                                    float* __restrict__ part_lse) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nth = (int64_t)gridDim.x * blockDim.x;
  auto prefix_of = [&](int s) -> int {  // prefix tokens of sequence s (0: no group)
    const int g = seq_group[s];
    if (g < 0) return 0;
    if (g >= num_groups) {
      flag_error(PA_DEVERR_QLEN_RANGE);
      return 0;
    }
    return prefix_lens[g];
  };
  // suffix views
  for (int64_t i = tid; i < (int64_t)S * max_blocks; i += nth) {
    const int s = (int)(i / max_blocks), b = (int)(i % max_blocks);
    const int pb = prefix_of(s) / kBlock;
    suffix_bt[i] = b + pb < max_blocks ? block_tables[(int64_t)s * max_blocks + b + pb] : 0;
    if (b == 0) {
      const int p = prefix_of(s), c = context_lens[s];
      if (p < 0 || p % kBlock != 0 || p > c || p > max_prefix_blocks * kBlock) {
        flag_error(PA_DEVERR_CONTEXT_RANGE);
        suffix_cl[s] = 0;
      } else {
        suffix_cl[s] = c - p;
      }
      // a grouped sequence must be listed among its group's (sorted) members
      const int g = seq_group[s];
      if (g >= 0 && g < num_groups) {
        int lo = cu_group[g], hi = cu_group[g + 1] - 1;
        bool found = false;
        while (lo <= hi && lo >= 0 && hi < num_members) {
          const int mid = (lo + hi) >> 1, v = group_members[mid];
          if (v == s) {
            found = true;
            break;
          }
          if (v < s) lo = mid + 1; else hi = mid - 1;
        }
        if (!found) flag_error(PA_DEVERR_QLEN_RANGE);
      }
    }
  }
  // gathered member queries: Hq * D bf16 = Hq * 16 uint4 per member
  const int per = Hq * (kHeadDim * 2 / 16);
  for (int64_t i = tid; i < (int64_t)num_members * per; i += nth) {
    const int m = (int)(i / per), k = (int)(i % per);
    const int s = group_members[m];
    if (s < 0 || s >= S) {
      if (k == 0) flag_error(PA_DEVERR_QLEN_RANGE);
      q_g[i] = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    q_g[i] = q[(int64_t)s * per + k];
  }
  // prefix block tables and the membership check
  for (int64_t i = tid; i < (int64_t)num_groups * max_prefix_blocks; i += nth) {
    const int g = (int)(i / max_prefix_blocks), b = (int)(i % max_prefix_blocks);
    const int m0 = cu_group[g], m1 = cu_group[g + 1];
    const int pb = prefix_lens[g] / kBlock;
    int id = 0;
    if (m0 < m1 && m0 >= 0 && m0 < num_members && b < pb && b < max_blocks) {
      const int s = group_members[m0];
      if (s >= 0 && s < S) id = block_tables[(int64_t)s * max_blocks + b];
    }
    prefix_bt[i] = id;
    if (b == 0 && (m0 < 0 || m1 < m0 || m1 > num_members || prefix_lens[g] <= 0))
      flag_error(PA_DEVERR_QLEN_RANGE);
  }
  // every listed member belongs to the group whose range holds it, once, in
  // increasing order (one thread per member; its group by binary search)
  for (int64_t m = tid; m < num_members; m += nth) {
    int lo = 0, hi = num_groups - 1, g = -1;
    while (lo <= hi) {  // the group g with cu_group[g] <= m < cu_group[g + 1]
      const int mid = (lo + hi) >> 1;
      if (cu_group[mid + 1] <= m) lo = mid + 1;
      else if (cu_group[mid] > m) hi = mid - 1;
      else { g = mid; break; }
    }
    const int s = group_members[m];
    if (g < 0 || s < 0 || s >= S || seq_group[s] != g ||
        (m > cu_group[g] && group_members[m - 1] >= s))
      flag_error(PA_DEVERR_QLEN_RANGE);
  }
  // empty prefix partial (0, -inf) for every sequence in no group
  const int per_row = kHeadDim / 4;
  for (int64_t i = tid; i < (int64_t)S * Hq * per_row; i += nth) {
    const int64_t row = i / per_row;  // s * Hq + h
    const int s = (int)(row / Hq);
    if (seq_group[s] >= 0) continue;
    reinterpret_cast<float4*>(part_o + (row * 2) * kHeadDim)[i % per_row] =
        make_float4(0.f, 0.f, 0.f, 0.f);
    if (i % per_row == 0) part_lse[row * 2] = neg_inf();
  }
}

}  // namespace

unsigned take_error_word_cascade(cudaStream_t stream, int* rc) {
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

extern "C" size_t pa_decode_cascade_workspace_size(const pa_shape* shape, int num_groups,
                                                   int num_members, int max_group_size,
                                                   int max_prefix_len) {
  if (check_shape_common(shape) != PA_OK) return 0;
  CascadeLayout L;
  if (cascade_layout(shape, num_groups, num_members, max_group_size, max_prefix_len, &L) !=
      PA_OK)
    return 0;
  return L.total;
}

extern "C" int pa_decode_cascade_ex(const pa_bf16* q, const pa_bf16* k_cache,
                                    const pa_bf16* v_cache, const int32_t* block_tables,
                                    const int32_t* context_lens, const int32_t* seq_group,
                                    int num_groups, const int32_t* cu_group,
                                    const int32_t* group_members, const int32_t* prefix_lens,
                                    int num_members, int max_group_size, int max_prefix_len,
                                    float scale, pa_bf16* out, float* lse,
                                    const pa_shape* shape, int policy, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  pa::NvtxRange nvtx_range("pa_decode_cascade");
  if (policy != PA_CASCADE_AUTO && policy != PA_CASCADE_ALWAYS && policy != PA_CASCADE_PLAIN)
    return PA_ERR_ARG;
  int rc = check_shape_common(shape);
  if (rc != PA_OK) return rc;
  const int S = shape->num_seqs;
  if (S == 0) return PA_OK;
  if (shape->num_q_heads != 2 * shape->num_kv_heads) return PA_ERR_UNSUPPORTED;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !seq_group || !out)
    return PA_ERR_ARG;
  if (num_groups > 0 && (!cu_group || !group_members || !prefix_lens)) return PA_ERR_ARG;
  if (num_members > 0 && num_groups <= 0) return PA_ERR_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || (lse && !aligned(lse, 4))) return PA_ERR_ARG;
  CascadeLayout L;
  rc = cascade_layout(shape, num_groups, num_members, max_group_size, max_prefix_len, &L);
  if (rc != PA_OK) return rc;
  if (!workspace || workspace_bytes < L.total || !aligned(workspace, 256))
    return PA_ERR_WORKSPACE;
  if (policy == PA_CASCADE_PLAIN ||
      (policy == PA_CASCADE_AUTO &&
       !cascade_pays(shape, num_groups, num_members, max_prefix_len)))
    return pa_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, lse, shape, 0,
                     workspace, workspace_bytes, stream);
  char* ws = static_cast<char*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  pa_bf16* q_g = reinterpret_cast<pa_bf16*>(ws + L.q_g);
  int32_t* prefix_bt = reinterpret_cast<int32_t*>(ws + L.prefix_bt);
  int32_t* suffix_bt = reinterpret_cast<int32_t*>(ws + L.suffix_bt);
  int32_t* suffix_cl = reinterpret_cast<int32_t*>(ws + L.suffix_cl);
  float* part_o = reinterpret_cast<float*>(ws + L.part_o);
  float* part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  const int Hq = shape->num_q_heads;

  DeviceInfo dev;
  if (!current_device_info(&dev)) return PA_ERR_CUDA;
  if (launch_dependent(cascade_prep_kernel, dim3(2 * dev.num_sms), dim3(256), 0, st,
                       reinterpret_cast<const uint4*>(q), block_tables, context_lens, seq_group,
                       cu_group, group_members, prefix_lens, S, Hq, shape->max_blocks_per_seq,
                       num_groups, num_members, max_prefix_len / kBlock,
                       reinterpret_cast<uint4*>(q_g), prefix_bt, suffix_bt, suffix_cl, part_o,
                       part_lse) != cudaSuccess)
    return PA_ERR_CUDA;
  // prefix half: slot 0 of each member's rows
  RowsOut prefix_rows;
  prefix_rows.o = part_o;
  prefix_rows.lse = part_lse;
  prefix_rows.stride = 2;
  prefix_rows.slot = 0;
  prefix_rows.tokens = S;
  // Order on the stream: prep -> prefix attention (tc_ctas CTAs) -> suffix
  // decode, launched while the prefix grid runs and sized for the other SMs;
  // it waits for the prefix grid only on its way out -> suffix merge ->
  // prefix merge -> the two-way merge. Every wait in that chain implies the
  // completion of the grids before it.
  if (L.tg.enabled) {
    rc = launch_prefill_tc(L.tg, q_g, k_cache, v_cache, prefix_bt, prefix_lens, cu_group,
                           num_members, /*causal=*/0, scale, nullptr, nullptr, &L.tc_shape,
                           ws + L.tc_ws, st, /*min_q_len=*/1, &prefix_rows, group_members,
                           /*parts=*/1);
    if (rc != PA_OK) return rc;
  }
  // suffix half: slot 1 of every row
  RowsOut suffix_rows = prefix_rows;
  suffix_rows.slot = 1;
  rc = decode_rows(q, k_cache, v_cache, suffix_bt, suffix_cl, scale, &L.suffix_shape,
                   suffix_rows, ws + L.dec_ws, L.dec_ws_bytes, st, L.tg.enabled ? 1 : 0,
                   L.suffix_sms);
  if (rc != PA_OK) return rc;
  if (L.tg.enabled) {
    rc = launch_prefill_tc(L.tg, q_g, k_cache, v_cache, prefix_bt, prefix_lens, cu_group,
                           num_members, /*causal=*/0, scale, nullptr, nullptr, &L.tc_shape,
                           ws + L.tc_ws, st, /*min_q_len=*/1, &prefix_rows, group_members,
                           /*parts=*/2);
    if (rc != PA_OK) return rc;
  }
  return pa_splitk_reduce(part_o, part_lse, S, Hq, 2, kHeadDim, out, lse, stream);
}

extern "C" int pa_decode_cascade(const pa_bf16* q, const pa_bf16* k_cache,
                                 const pa_bf16* v_cache, const int32_t* block_tables,
                                 const int32_t* context_lens, const int32_t* seq_group,
                                 int num_groups, const int32_t* cu_group,
                                 const int32_t* group_members, const int32_t* prefix_lens,
                                 int num_members, int max_group_size, int max_prefix_len,
                                 float scale, pa_bf16* out, float* lse, const pa_shape* shape,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  return pa_decode_cascade_ex(q, k_cache, v_cache, block_tables, context_lens, seq_group,
                              num_groups, cu_group, group_members, prefix_lens, num_members,
                              max_group_size, max_prefix_len, scale, out, lse, shape,
                              PA_CASCADE_AUTO, workspace, workspace_bytes, stream);
}
