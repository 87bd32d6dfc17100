// C-ABI host library: argument checks, workspace ownership, tensor maps and
// the launch sequence of the forward pass. See include/moe.h for the contract.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

using namespace moe;

namespace {

thread_local char g_msg[512] = "";

moe_status fail(moe_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return s;
}

moe_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define CUDA_TRY(call)                                   \
  do {                                                   \
    cudaError_t _e = (call);                             \
    if (_e != cudaSuccess) return cuda_fail(_e, #call);  \
  } while (0)

constexpr int kMaxTile = 256;       // largest tile_m the sort accepts

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int fmt_of_adtype(int a) { return a == MOE_A_BF16 ? FMT_F16 : (a == MOE_A_FP8 ? FMT_E4M3 : FMT_E2M1); }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Host-side fault injection (moe_debug_inject): the index of the workspace
// allocation the next moe_create fails, or -1. One-shot.
std::atomic<long> g_fail_alloc{-1};

}  // namespace

void moe::set_last_error_message(const char* msg) { snprintf(g_msg, sizeof(g_msg), "%s", msg); }

struct moe_ctx {
  int H, I, E, K, max_tokens, device, num_sms;
  long cap_rows, cap_blocks;
  int hist_chunks;
  int32_t *sorted_ids, *block_expert, *expert_count, *expert_offset, *active_experts, *meta, *hist;
  uint8_t *xq, *xs, *inter_q, *inter_s;
  uint8_t *xq_sorted, *xs_sorted;  // tensor-core path: activations in sorted order + chunked scales
  int32_t* pair_row;
  int32_t* row_tok;  // few-rows path: token and top-k weight of every sorted row
  float* row_w;
  int4* active_info;
  float* acc32;
  int* err;
  void* st_x;
  int32_t* st_ids;
  float* st_w;
  void* st_out;
  // tcgen05 family maps (keyed by pointer and kind)
  const void* tm_w13tc_key; int tm_w13tc_kind; CUtensorMap tm_w13tc;
  const void* tm_w2tc_key; int tm_w2tc_kind; CUtensorMap tm_w2tc;
  const void* tm_w13sw_key; int tm_w13sw_kind; CUtensorMap tm_w13sw;  // 128-row gate / up tiles
  const void* tm_w2sw_key; CUtensorMap tm_w2sw;  // packed w2, 64-byte rows (few-rows stage 2)
  int last_inter_stride;
  int tc_min_rows;  // mean routed rows per active expert from which the tcgen05 path is used
  int tc_group;     // many-rows stage 2: N tiles per group of the tile order (0: chosen per call)
  int fused;        // 1: sort + scatter in one launch (calls of up to SORT_SMALL_MAX_PAIRS pairs)
  int split_k;      // 1: few-rows stage 1 splits K over clusters when its units fill few SMs
  int split_cap[3][4];  // [kind][ks]: clusters of the split stage-1 kernel resident at once (0: unknown)
  // prepacked stage-2 weights (moe_prepack): used when moe_forward's w2 is pk_src
  const uint8_t* pk_src;
  int pk_adt;  // the a_dtype whose few-rows stage 2 the packed copy serves
  uint8_t* pk_codes;
  uint8_t* pk_scales;
  const void* tm_w2pk_key; int tm_w2pk_kind; CUtensorMap tm_w2pk;
  int last_inter_layout;
  int last_tile_m;
  // profiling (moe_set_profiling)
  int profiling;
  cudaEvent_t ev[8];
  const char* ev_name[8];
  int ev_n;
};

static void prof_mark(moe_ctx* c, cudaStream_t st, const char* name) {
  if (!c->profiling || c->ev_n >= 7) return;
  cudaEventRecord(c->ev[c->ev_n], st);
  c->ev_name[c->ev_n] = name;
  ++c->ev_n;
}

static void free_ctx(moe_ctx* c) {
  void* ptrs[] = {c->sorted_ids, c->block_expert, c->expert_count, c->expert_offset, c->active_experts,
                  c->meta, c->hist, c->xq, c->xs, c->inter_q, c->inter_s, c->acc32, c->err,
                  c->xq_sorted, c->xs_sorted, c->pair_row, c->row_tok, c->row_w, c->active_info,
                  c->st_x, c->st_ids, c->st_w, c->st_out};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  for (cudaEvent_t e : c->ev)
    if (e) cudaEventDestroy(e);
  delete c;
}

static moe_status encode(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
                         const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swz, const char* what) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(m, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed: %d", what, (int)r);
  return MOE_OK;
}

// fp4 weights for the tcgen05 kinds: mxf8f6f4 reads e2m1 as one 16-element
// group per 16 bytes of shared memory (TMA type 16U4_ALIGN16B expands the
// packed rows); mxf4 reads them packed (plain bytes).
static moe_status make_w13tc_map(moe_ctx* c, const uint8_t* w13, int kind) {
  if (c->tm_w13tc_key == w13 && c->tm_w13tc_kind == kind) return MOE_OK;
  const cuuint64_t H = c->H, I = c->I, E = c->E;
  cuuint64_t strides[3] = {H / 2, I * H / 2, 2 * I * H / 2};
  moe_status s;
  if (kind == TC_A8W4) {
    cuuint64_t dims[4] = {H, I, 2, E};
    cuuint32_t box[4] = {128, 64, 1, 1};
    s = encode(&c->tm_w13tc, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 4, w13, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, "w13 fp4 unpacked");
  } else {
    cuuint64_t dims[4] = {H / 2, I, 2, E};
    cuuint32_t box[4] = {128, 64, 1, 1};
    s = encode(&c->tm_w13tc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, w13, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, "w13 fp4 packed");
  }
  if (s != MOE_OK) return s;
  c->tm_w13tc_key = w13;
  c->tm_w13tc_kind = kind;
  return MOE_OK;
}

// Packed w2 in 64-byte rows (K tile 128, 64-byte swizzle) for the few-rows mxf4
// stage 2, whose K = inter is too short for 128-byte boxes to be filled.
static moe_status make_w2sw_map(moe_ctx* c, const uint8_t* w2) {
  if (c->tm_w2sw_key == w2) return MOE_OK;
  const cuuint64_t H = c->H, I = c->I, E = c->E;
  cuuint64_t dims[3] = {I / 2, H, E};
  cuuint64_t strides[2] = {I / 2, H * I / 2};
  cuuint32_t box[3] = {64, 128, 1};
  moe_status s = encode(&c->tm_w2sw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, w2, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_64B, "w2 fp4 packed, 64-byte rows");
  if (s != MOE_OK) return s;
  c->tm_w2sw_key = w2;
  return MOE_OK;
}

static moe_status make_w2tc_map(moe_ctx* c, const uint8_t* w2, int kind) {
  if (c->tm_w2tc_key == w2 && c->tm_w2tc_kind == kind) return MOE_OK;
  const cuuint64_t H = c->H, I = c->I, E = c->E;
  cuuint64_t strides[2] = {I / 2, H * I / 2};
  cuuint32_t box[3] = {128, 128, 1};
  moe_status s;
  if (kind == TC_A8W4) {
    cuuint64_t dims[3] = {I, H, E};
    s = encode(&c->tm_w2tc, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, w2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, "w2 fp4 unpacked");
  } else {
    cuuint64_t dims[3] = {I / 2, H, E};
    s = encode(&c->tm_w2tc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, w2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, "w2 fp4 packed");
  }
  if (s != MOE_OK) return s;
  c->tm_w2tc_key = w2;
  c->tm_w2tc_kind = kind;
  return MOE_OK;
}

// Stage-1 weights of the few-rows tensor-core path: 128 gate (or up) rows per box.
static moe_status make_w13sw_map(moe_ctx* c, const uint8_t* w13, int kind) {
  if (c->tm_w13sw_key == w13 && c->tm_w13sw_kind == kind) return MOE_OK;
  const cuuint64_t H = c->H, I = c->I, E = c->E;
  cuuint64_t strides[3] = {H / 2, I * H / 2, 2 * I * H / 2};
  cuuint32_t box[4] = {128, 128, 1, 1};
  moe_status s;
  if (kind == TC_A8W4) {
    cuuint64_t dims[4] = {H, I, 2, E};
    s = encode(&c->tm_w13sw, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 4, w13, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, "w13 fp4 unpacked, 128 rows");
  } else {
    cuuint64_t dims[4] = {H / 2, I, 2, E};
    s = encode(&c->tm_w13sw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, w13, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, "w13 fp4 packed, 128 rows");
  }
  if (s != MOE_OK) return s;
  c->tm_w13sw_key = w13;
  c->tm_w13sw_kind = kind;
  return MOE_OK;
}

// Prepacked w2 (kernels_pack.cu): rows of 64 bytes (one 128-element K chunk), each
// 128 consecutive rows one (expert, 128-row tile, K chunk) block; unpacked by TMA
// to 128-byte rows for kind::mxf8f6f4.
static moe_status make_w2pk_map(moe_ctx* c, int kind) {
  if (c->tm_w2pk_key == c->pk_codes && c->tm_w2pk_kind == kind) return MOE_OK;
  const cuuint64_t rows = (cuuint64_t)c->E * (c->H / 128) * (c->I / 128) * 128;
  cuuint64_t strides[1] = {64};
  moe_status s;
  if (kind == TC_A8W4) {
    cuuint64_t dims[2] = {128, rows};
    cuuint32_t box[2] = {128, 128};
    s = encode(&c->tm_w2pk, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, c->pk_codes, dims, strides, box,
               CU_TENSOR_MAP_SWIZZLE_128B, "prepacked w2, unpacked");
  } else {
    cuuint64_t dims[2] = {64, rows};
    cuuint32_t box[2] = {64, 128};
    s = encode(&c->tm_w2pk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, c->pk_codes, dims, strides, box,
               CU_TENSOR_MAP_SWIZZLE_64B, "prepacked w2");
  }
  if (s != MOE_OK) return s;
  c->tm_w2pk_key = c->pk_codes;
  c->tm_w2pk_kind = kind;
  return MOE_OK;
}

static SortOut sort_out(moe_ctx* c) {
  SortOut so;
  so.sorted_ids = c->sorted_ids;
  so.block_expert = c->block_expert;
  so.expert_count = c->expert_count;
  so.expert_offset = c->expert_offset;
  so.active_experts = c->active_experts;
  so.meta = c->meta;
  return so;
}

static void fill_sort_view(moe_ctx* c, int tile_m, moe_sort_view* v) {
  v->sorted_ids = c->sorted_ids;
  v->block_expert = c->block_expert;
  v->expert_count = c->expert_count;
  v->expert_offset = c->expert_offset;
  v->active_experts = c->active_experts;
  v->meta = c->meta;
  v->tile_m = tile_m;
  v->max_rows = c->cap_rows;
  v->max_blocks = c->cap_blocks;
}

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_OOM: return "out of device memory";
    case MOE_ERR_BAD_EXPERT_ID: return "expert id out of range (pairs dropped)";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

const char* moe_last_error_message(void) { return g_msg; }

moe_status moe_create(moe_ctx** out, int H, int I, int E, int K, int max_tokens, int device) {
  if (!out) return fail(MOE_ERR_INVALID_ARG, "ctx out-pointer is NULL");
  *out = nullptr;
  if (H <= 0 || I <= 0 || E <= 0 || K <= 0 || max_tokens <= 0)
    return fail(MOE_ERR_INVALID_ARG, "sizes must be positive (H=%d I=%d E=%d K=%d max_tokens=%d)", H, I, E, K, max_tokens);
  if (H % 128 || I % 128) return fail(MOE_ERR_UNSUPPORTED, "hidden and inter must be multiples of 128");
  if (H > 16384 || I > 16384) return fail(MOE_ERR_UNSUPPORTED, "hidden and inter are limited to 16384");
  if (E > SORT_MAX_EXPERTS) return fail(MOE_ERR_UNSUPPORTED, "num_experts is limited to %d", SORT_MAX_EXPERTS);
  if ((long)max_tokens * K > (1L << 30)) return fail(MOE_ERR_UNSUPPORTED, "max_tokens * topk too large");
  int ndev = 0;
  CUDA_TRY(cudaGetDeviceCount(&ndev));
  if (device < 0 || device >= ndev) return fail(MOE_ERR_INVALID_ARG, "device %d out of range (%d devices)", device, ndev);
  cudaDeviceProp prop;
  CUDA_TRY(cudaGetDeviceProperties(&prop, device));
  if (prop.major != 10 || prop.minor != 3)
    return fail(MOE_ERR_UNSUPPORTED, "needs a compute capability 10.3 GPU (GB300), device %d is %d.%d", device,
                prop.major, prop.minor);
  CUDA_TRY(cudaSetDevice(device));

  moe_ctx* c = new moe_ctx();
  std::memset(c, 0, sizeof(*c));
  c->H = H; c->I = I; c->E = E; c->K = K; c->max_tokens = max_tokens; c->device = device;
  c->num_sms = prop.multiProcessorCount;
  long pairs = (long)max_tokens * K;
  c->cap_rows = pairs + (long)(E < pairs ? E : pairs) * (kMaxTile - 1);
  c->cap_rows = (c->cap_rows + kMaxTile - 1) / kMaxTile * kMaxTile;
  c->cap_blocks = c->cap_rows;  // enough for tile_m = 1
  c->hist_chunks = (int)((pairs + SORT_CHUNK - 1) / SORT_CHUNK);
  if (c->hist_chunks < 1) c->hist_chunks = 1;

  struct { void** p; size_t bytes; } allocs[] = {
      {(void**)&c->sorted_ids, sizeof(int32_t) * c->cap_rows},
      {(void**)&c->block_expert, sizeof(int32_t) * c->cap_blocks},
      {(void**)&c->expert_count, sizeof(int32_t) * E},
      {(void**)&c->expert_offset, sizeof(int32_t) * (E + 1)},
      {(void**)&c->active_experts, sizeof(int32_t) * E},
      {(void**)&c->meta, sizeof(int32_t) * META_WORDS},
      {(void**)&c->hist, sizeof(int32_t) * (size_t)c->hist_chunks * E},
      {(void**)&c->xq, (size_t)max_tokens * H * 2},
      {(void**)&c->xs, (size_t)max_tokens * scale_row_stride(H)},
      {(void**)&c->inter_q, (size_t)c->cap_rows * (A16_TERMS * I / 2 > 2 * I ? A16_TERMS * I / 2 : 2 * I)},
      {(void**)&c->inter_s, (size_t)c->cap_rows * A16_TERMS * scale_row_stride(I)},
      {(void**)&c->acc32, sizeof(float) * (size_t)max_tokens * H},
      {(void**)&c->xq_sorted, (size_t)c->cap_rows * A16_TERMS * H / 2},
      {(void**)&c->xs_sorted, (size_t)c->cap_rows * A16_TERMS * scale_row_stride(H)},
      {(void**)&c->pair_row, sizeof(int32_t) * pairs},
      {(void**)&c->row_tok, sizeof(int32_t) * c->cap_rows},
      {(void**)&c->row_w, sizeof(float) * c->cap_rows},
      {(void**)&c->active_info, sizeof(int4) * E},
      {(void**)&c->err, sizeof(int) * 4},
      {(void**)&c->st_x, (size_t)max_tokens * H * 2},
      {(void**)&c->st_ids, sizeof(int32_t) * pairs},
      {(void**)&c->st_w, sizeof(float) * pairs},
      {(void**)&c->st_out, (size_t)max_tokens * H * 2},
  };
  const long inject = g_fail_alloc.exchange(-1);
  long idx = 0;
  for (auto& a : allocs) {
    cudaError_t e = idx == inject ? cudaErrorMemoryAllocation : cudaMalloc(a.p, a.bytes);
    if (e != cudaSuccess) {
      cudaGetLastError();
      free_ctx(c);  // releases every buffer allocated so far
      return fail(MOE_ERR_OOM, "cudaMalloc(%zu) failed%s: %s", a.bytes, idx == inject ? " (injected)" : "",
                  cudaGetErrorString(e));
    }
    ++idx;
  }
  cudaError_t e = cudaMemset(c->err, 0, sizeof(int) * 4);
  if (e == cudaSuccess) e = cudaMemset(c->meta, 0, sizeof(int32_t) * META_WORDS);
  if (e == cudaSuccess) e = prep_set_smem_limits();
  if (e == cudaSuccess) e = tc_set_smem_limits();
  if (e == cudaSuccess) e = swap_set_smem_limits();
  if (e != cudaSuccess) {
    free_ctx(c);
    return cuda_fail(e, "context setup");
  }
  c->tc_min_rows = 32;
  if (const char* v = getenv("MOE_TC_MIN_ROWS")) c->tc_min_rows = atoi(v);
  if (const char* v = getenv("MOE_TC_GROUP")) c->tc_group = atoi(v);
  c->fused = 0;
  if (const char* v = getenv("MOE_FUSED")) c->fused = atoi(v);
  c->split_k = 1;
  if (const char* v = getenv("MOE_SPLITK")) c->split_k = atoi(v);
  c->last_inter_stride = scale_row_stride(I);
  *out = c;
  return MOE_OK;
}

moe_status moe_destroy(moe_ctx* c) {
  if (!c) return MOE_OK;
  cudaSetDevice(c->device);
  cudaDeviceSynchronize();
  free_ctx(c);
  return MOE_OK;
}

moe_status moe_get_workspace(moe_ctx* c, moe_workspace_view* v) {
  if (!c || !v) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
  fill_sort_view(c, c->last_tile_m, &v->sort);
  v->act_codes = c->xq;
  v->act_scales = c->xs;
  v->inter_codes = c->inter_q;
  v->inter_scales = c->inter_s;
  v->acc32 = c->acc32;
  v->act_scale_stride = scale_row_stride(c->H);
  v->inter_scale_stride = c->last_inter_stride;
  v->inter_scale_layout = c->last_inter_layout;
  v->act_sorted_codes = c->xq_sorted;
  v->act_sorted_scales = c->xs_sorted;
  v->act_sorted_scale_stride = scale_row_stride(c->H);
  v->a16_terms = A16_TERMS;
  return MOE_OK;
}

moe_status moe_sort(moe_ctx* c, const int32_t* ids, int T, int tile_m, moe_sort_view* out, void* stream) {
  if (!c || !out) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
  if (T < 0 || T > c->max_tokens) return fail(MOE_ERR_INVALID_ARG, "num_tokens %d outside [0, %d]", T, c->max_tokens);
  if (tile_m < 1 || tile_m > kMaxTile || (tile_m & (tile_m - 1)))
    return fail(MOE_ERR_INVALID_ARG, "tile_m must be a power of two in [1, %d]", kMaxTile);
  if (T > 0 && !ids) return fail(MOE_ERR_INVALID_ARG, "topk_ids is NULL");
  CUDA_TRY(cudaSetDevice(c->device));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_sort(ids, (long)T * c->K, c->E, tile_m, sort_out(c), c->hist, c->hist_chunks, c->err, st);
  if (e != cudaSuccess) return cuda_fail(e, "sort launch");
  c->last_tile_m = tile_m;
  fill_sort_view(c, tile_m, out);
  return MOE_OK;
}

}  // extern "C"

// The forward pass behind moe_forward. out == nullptr: no finalize, the fp32 sums
// stay in c->acc32 (the expert-parallel emulation reads them); neg_masked: negative
// expert ids mean "no expert here" (skipped, not flagged).
static moe_status forward_impl(moe_ctx* c, const void* x, const int32_t* ids, const float* w, int T,
                               const uint8_t* w13, const uint8_t* w13s, const uint8_t* w2, const uint8_t* w2s, int act,
                               float beta, float lbeta, int adt, void* out, void* stream, bool neg_masked) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "ctx is NULL");
  if (T < 0 || T > c->max_tokens) return fail(MOE_ERR_INVALID_ARG, "num_tokens %d outside [0, %d]", T, c->max_tokens);
  if (act != MOE_ACT_SILU && act != MOE_ACT_SITUV2) return fail(MOE_ERR_UNSUPPORTED, "activation %d is not silu or situv2", act);
  if (adt != MOE_A_BF16 && adt != MOE_A_FP8 && adt != MOE_A_FP4) return fail(MOE_ERR_UNSUPPORTED, "a_dtype %d unknown", adt);
  if (act == MOE_ACT_SITUV2 && !(beta > 0.0f && lbeta > 0.0f && beta < 3e38f && lbeta < 3e38f))
    return fail(MOE_ERR_INVALID_ARG, "SiTUv2 needs finite beta > 0 and linear_beta > 0");
  if (T == 0) return MOE_OK;
  const void* ptrs[] = {x, ids, w, w13, w13s, w2, w2s, out ? out : x};
  for (const void* p : ptrs) {
    if (!p) return fail(MOE_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned16(p)) return fail(MOE_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  }
  CUDA_TRY(cudaSetDevice(c->device));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int fmt = fmt_of_adtype(adt);
  const long pairs = (long)T * c->K;
  const long max_active = pairs < c->E ? pairs : c->E;
  // Path: the many-rows tcgen05 kernels (128 routed rows x 128 weight rows per
  // tile) once the mean number of routed rows per active expert reaches
  // tc_min_rows (fp8 / fp4 activations); below that the few-rows tcgen05
  // kernels (128 weight rows x up to 64 routed rows per MMA).
  const bool use_tc = adt != MOE_A_BF16 && c->tc_min_rows > 0 && pairs >= (long)c->tc_min_rows * max_active &&
                      c->H <= TC_MAX_K && c->I <= TC_MAX_K;
  const bool use_sw = !use_tc;
  const bool use_packed = use_sw && c->pk_codes && c->pk_src == w2 && c->pk_adt == adt;
  const int tile_m = use_tc ? TC_TILE_M : 1;
  const int kind = adt == MOE_A_FP8 ? TC_A8W4 : TC_A4W4;
  const int swkind = adt == MOE_A_BF16 ? SW_A16 : (adt == MOE_A_FP8 ? SW_A8 : SW_A4);
  const int wkind = adt == MOE_A_FP8 ? TC_A8W4 : TC_A4W4;  // weight map type: unpacked for mxf8f6f4, packed for mxf4
  // few-rows path: sub-rows per sorted row (bf16: A16_TERMS e2m1 code terms), bytes per
  // sub-row of the sorted activations / intermediate, and their scale strides
  const int subs = adt == MOE_A_BF16 ? A16_TERMS : 1;
  const int x_row = adt == MOE_A_FP8 ? c->H : c->H / 2;
  const int i_row = adt == MOE_A_FP8 ? c->I : c->I / 2;
  const int xs_sw = scale_row_stride(c->H);
  const int is_sw = scale_row_stride(c->I);
  CUtensorMap tm_inter, tm_xs;
  moe_status ms;
  if (use_tc) {
    ms = make_w13tc_map(c, w13, kind);
    if (ms != MOE_OK) return ms;
    ms = make_w2tc_map(c, w2, kind);
    if (ms != MOE_OK) return ms;
    const cuuint64_t irow = adt == MOE_A_FP8 ? (cuuint64_t)c->I : (cuuint64_t)c->I / 2;
    cuuint64_t idims[2] = {irow, (cuuint64_t)c->cap_rows}, istr[1] = {irow};
    cuuint32_t ibox[2] = {128, 128};
    ms = encode(&tm_inter, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, c->inter_q, idims, istr, ibox, CU_TENSOR_MAP_SWIZZLE_128B, "intermediate");
    if (ms != MOE_OK) return ms;
    const cuuint64_t xrow = adt == MOE_A_FP8 ? (cuuint64_t)c->H : (cuuint64_t)c->H / 2;
    cuuint64_t xdims[2] = {xrow, (cuuint64_t)c->cap_rows}, xstr[1] = {xrow};
    ms = encode(&tm_xs, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, c->xq_sorted, xdims, xstr, ibox, CU_TENSOR_MAP_SWIZZLE_128B, "sorted activations");
    if (ms != MOE_OK) return ms;
  } else {
    ms = make_w13sw_map(c, w13, wkind);
    if (ms != MOE_OK) return ms;
    // stage 2 streams K = inter in the kernel's row width: 64-byte rows take the
    // packed 64-byte-box map, 128-byte rows the 128-byte one (unpacked for A8);
    // a prepacked copy of these weights takes its own map
    const bool narrow2 = swap_row_bytes(swkind, 2) == 64;
    if (use_packed) {
      ms = make_w2pk_map(c, wkind);
    } else {
      ms = narrow2 ? make_w2sw_map(c, w2) : make_w2tc_map(c, w2, wkind);
    }
    if (ms != MOE_OK) return ms;
    cuuint32_t box[2] = {128, 16};
    cuuint32_t ibox[2] = {narrow2 ? 64u : 128u, 16};
    cuuint64_t idims[2] = {(cuuint64_t)i_row, (cuuint64_t)c->cap_rows * subs}, istr[1] = {(cuuint64_t)i_row};
    ms = encode(&tm_inter, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, c->inter_q, idims, istr, ibox,
                narrow2 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, "intermediate rows");
    if (ms != MOE_OK) return ms;
    cuuint64_t xdims[2] = {(cuuint64_t)x_row, (cuuint64_t)c->cap_rows * subs}, xstr[1] = {(cuuint64_t)x_row};
    ms = encode(&tm_xs, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, c->xq_sorted, xdims, xstr, box, CU_TENSOR_MAP_SWIZZLE_128B, "sorted activation rows");
    if (ms != MOE_OK) return ms;
  }

  c->ev_n = 0;
  SortOut so = sort_out(c);
  so.pair_row = c->pair_row;
  so.neg_masked = neg_masked ? 1 : 0;
  if (use_sw) so.active_info = c->active_info;
  c->last_tile_m = tile_m;
  c->last_inter_layout = use_tc ? 1 : (adt == MOE_A_BF16 ? 2 : 0);
  c->last_inter_stride = use_sw ? is_sw : scale_row_stride(c->I);
  ScatterOut sc{};
  sc.codes = c->xq_sorted;
  sc.scales = c->xs_sorted;
  sc.sstride = use_tc ? 0 : xs_sw;
  sc.acc32 = c->acc32;
  if (use_sw) {
    sc.topk_w = w;
    sc.row_tok = c->row_tok;
    sc.row_w = c->row_w;
  }
  cudaError_t e;
  const bool one_launch = c->fused && pairs <= SORT_SMALL_MAX_PAIRS;  // sort + scatter fused
  if (one_launch) {
    prof_mark(c, st, "sort+act_quant");
    e = launch_sort_scatter(ids, pairs, c->E, tile_m, so, c->err, x, T, c->H, c->K, swkind, sc, c->num_sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "sort + activation scatter launch");
  } else {
    prof_mark(c, st, "sort");
    e = launch_sort(ids, pairs, c->E, tile_m, so, c->hist, c->hist_chunks, c->err, st);
    if (e != cudaSuccess) return cuda_fail(e, "sort launch");
    prof_mark(c, st, "act_quant");
    e = launch_act_scatter(x, T, c->H, c->K, swkind, c->pair_row, sc, c->num_sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "activation quantisation launch");
  }

  StageParams p{};
  p.sorted_ids = c->sorted_ids;
  p.block_expert = c->block_expert;
  p.expert_offset = c->expert_offset;
  p.expert_count = c->expert_count;
  p.active_experts = c->active_experts;
  p.active_info = c->active_info;
  p.meta = c->meta;
  p.T = T; p.H = c->H; p.I = c->I; p.E = c->E; p.K = c->K;
  p.act = act; p.beta = beta; p.lbeta = lbeta;
  p.err = c->err;

  const long max_blocks = (pairs + max_active * (tile_m - 1)) / tile_m;  // upper bound on sort blocks
  StageParams p1 = p;
  p1.aq = c->xq; p1.as = c->xs; p1.wscale = w13s;
  p1.oq = c->inter_q; p1.os = c->inter_s;
  p1.xs_stride = scale_row_stride(c->H);
  p1.os_stride = scale_row_stride(c->I);
  StageParams p2 = p;
  p2.aq = c->inter_q; p2.as = c->inter_s; p2.wscale = w2s;
  p2.acc32 = c->acc32; p2.topk_w = w;
  p2.xs_stride = scale_row_stride(c->I);

  if (use_tc) {
    long t1 = max_blocks * (c->I / 64), t2 = max_blocks * (c->H / 128);
    // Stage-2 tile order: block-major keeps each 128-row block of the intermediate in
    // L2 while its N tiles run, and scatters into the fp32 combine buffer; N tiles in
    // groups (the buffer's slice T x 128 x 4 bytes per N tile near 48 MB) keep the
    // buffer's active part in L2 but read the intermediate once per group. Groups pay
    // off when the buffer exceeds L2 and is larger than the intermediate they re-read.
    const double acc_bytes = (double)T * c->H * 4.0, slice = (double)T * 128 * 4.0;
    const double inter_bytes = (double)pairs * c->I * (adt == MOE_A_FP8 ? 1.0 + 1.0 / 32 : 0.5 + 1.0 / 32);
    const bool grouped = acc_bytes > 64.0 * (1 << 20) && acc_bytes > 2.0 * inter_bytes;
    p2.tile_group = grouped ? (int)(48.0 * (1 << 20) / slice) : 0;
    if (grouped && p2.tile_group < 1) p2.tile_group = 1;
    if (c->tc_group > 0) p2.tile_group = c->tc_group;
    prof_mark(c, st, "stage1");
    StageParams q1 = p1;
    q1.aq = c->xq_sorted;
    q1.as = c->xs_sorted;
    e = launch_tc_stage(kind, 1, q1, tm_xs, c->tm_w13tc, (int)(t1 < c->num_sms ? t1 : c->num_sms), st);
    if (e != cudaSuccess) return cuda_fail(e, "stage-1 launch");
    prof_mark(c, st, "stage2");
    e = launch_tc_stage(kind, 2, p2, tm_inter, c->tm_w2tc, (int)(t2 < c->num_sms ? t2 : c->num_sms), st);
    if (e != cudaSuccess) return cuda_fail(e, "stage-2 launch");
  } else {
    const long u2 = max_active * ((c->H + 255) / 256);
    StageParams q1 = p1;
    q1.aq = c->xq_sorted;
    q1.as = c->xs_sorted;
    q1.xs_stride = xs_sw;
    q1.os_stride = is_sw;
    prof_mark(c, st, "stage1");
    const long u1 = max_active * (c->I / 128);
    // split K over clusters of ks CTAs when the units leave most SMs idle (a few tokens)
    const int kt1 = c->H / (adt == MOE_A_FP8 ? 128 : 256);  // stage-1 K tiles
    // split only when one wave of resident clusters holds every unit (clusters need ks
    // free SMs of one GPC each, so fewer fit than num_sms / ks)
    auto cap = [&](int k) {
      if (!c->split_cap[swkind][k]) c->split_cap[swkind][k] = 1 + swap_split_max_clusters(swkind, k);
      return (long)c->split_cap[swkind][k] - 1;
    };
    // Also split in two when the units, taken in turn by persistent clusters of two
    // (each unit half as long), end in fewer rounds than on single CTAs: units just
    // above one SM each (T = 4: 186 units on 152 SMs take two rounds, on ~70 pairs
    // three half-length ones). Measured faster for bf16 and fp8 activations (TP8,
    // T = 4: 66.9 -> 63.6 and 76.8 -> 72.6 us) and slower for fp4 (50.2 -> 54.3 us),
    // whose items are shorter.
    int ks = 1;
    if (c->split_k && kt1 >= 3 && u1 <= cap(3)) ks = 3;
    else if (c->split_k && kt1 >= 2 && u1 <= cap(2)) ks = 2;
    else if (c->split_k && swkind != SW_A4 && kt1 >= 2 && cap(2) > 0) {
      const long r1 = (u1 + c->num_sms - 1) / c->num_sms, r2 = (u1 + cap(2) - 1) / cap(2);
      if (r2 < 2 * r1) ks = 2;
    }
    const long g1 = ks > 1 ? (u1 < cap(ks) ? u1 : cap(ks)) * ks : (u1 < c->num_sms ? u1 : c->num_sms);
    e = launch_swap_stage(swkind, 1, false, ks, q1, c->tm_w13sw, tm_xs, (int)g1, st);
    if (e != cudaSuccess) return cuda_fail(e, "stage-1 launch");
    StageParams q2 = p2;
    q2.xs_stride = is_sw;
    q2.row_tok = c->row_tok;
    q2.row_w = c->row_w;
    if (use_packed) {
      q2.wscale = c->pk_scales;
      q2.wpacked = c->pk_codes;
    }
    prof_mark(c, st, "stage2");
    e = launch_swap_stage(swkind, 2, use_packed, 1, q2,
                          use_packed ? c->tm_w2pk : (swap_row_bytes(swkind, 2) == 64 ? c->tm_w2sw : c->tm_w2tc),
                          tm_inter, (int)(u2 < c->num_sms ? u2 : c->num_sms), st);
    if (e != cudaSuccess) return cuda_fail(e, "stage-2 launch");
  }

  if (out) {
    prof_mark(c, st, "finalize");
    e = launch_finalize(c->acc32, (long)T * c->H, out, c->num_sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "finalize launch");
  }
  prof_mark(c, st, "end");
  return MOE_OK;
}

// ---------------------------------------------------------------------------
// Expert-parallel emulation (kernels_ep.cu)
// ---------------------------------------------------------------------------
struct moe_ep {
  int H, I, El, R, K, max_tokens, device, num_sms;
  moe_ctx* rank[EP_MAX_RANKS];
  void* recv_x;        // [R][max_tokens][H] bf16: the dispatch payload
  int32_t* recv_tok;   // [R][max_tokens]
  int32_t* recv_ids;   // [R][max_tokens][K] local expert ids, -1 for the pairs of other ranks
  float* recv_w;       // [R][max_tokens][K]
  int32_t* slot;       // [max_tokens][R] row of each token on each rank, -1 if not sent there
  int32_t* counts;     // [R] received tokens per rank (device)
  int32_t* counts_h;   // [R] (pinned host)
  uint8_t* wire_q;     // [R][max_tokens][H] e4m3: the combine payload
  uint8_t* wire_s;     // [R][max_tokens][H/32] e8m0
};

static void free_ep(moe_ep* p) {
  for (int r = 0; r < EP_MAX_RANKS; ++r)
    if (p->rank[r]) moe_destroy(p->rank[r]);
  void* ptrs[] = {p->recv_x, p->recv_tok, p->recv_ids, p->recv_w, p->slot, p->counts, p->wire_q, p->wire_s};
  for (void* q : ptrs)
    if (q) cudaFree(q);
  if (p->counts_h) cudaFreeHost(p->counts_h);
  delete p;
}

extern "C" {

moe_status moe_ep_create(moe_ep** out, int H, int I, int El, int R, int K, int max_tokens, int device) {
  if (!out) return fail(MOE_ERR_INVALID_ARG, "out-pointer is NULL");
  *out = nullptr;
  if (R < 1 || R > EP_MAX_RANKS) return fail(MOE_ERR_UNSUPPORTED, "ranks must be in [1, %d]", EP_MAX_RANKS);
  moe_ep* p = new moe_ep();
  std::memset(p, 0, sizeof(*p));
  p->H = H; p->I = I; p->El = El; p->R = R; p->K = K; p->max_tokens = max_tokens; p->device = device;
  for (int r = 0; r < R; ++r) {
    moe_status s = moe_create(&p->rank[r], H, I, El, K, max_tokens, device);
    if (s != MOE_OK) {
      free_ep(p);
      return s;
    }
  }
  p->num_sms = p->rank[0]->num_sms;
  const size_t rows = (size_t)R * max_tokens;
  struct { void** q; size_t bytes; } allocs[] = {
      {&p->recv_x, rows * H * 2},       {(void**)&p->recv_tok, rows * 4},     {(void**)&p->recv_ids, rows * K * 4},
      {(void**)&p->recv_w, rows * K * 4}, {(void**)&p->slot, rows * 4},       {(void**)&p->counts, (size_t)R * 4},
      {(void**)&p->wire_q, rows * H},   {(void**)&p->wire_s, rows * (H / 32)},
  };
  for (auto& a : allocs) {
    cudaError_t e = cudaMalloc(a.q, a.bytes);
    if (e != cudaSuccess) {
      cudaGetLastError();
      free_ep(p);
      return fail(MOE_ERR_OOM, "cudaMalloc(%zu) failed: %s", a.bytes, cudaGetErrorString(e));
    }
  }
  cudaError_t e = cudaMallocHost((void**)&p->counts_h, sizeof(int32_t) * R);
  if (e != cudaSuccess) {
    free_ep(p);
    return cuda_fail(e, "cudaMallocHost");
  }
  *out = p;
  return MOE_OK;
}

moe_status moe_ep_destroy(moe_ep* p) {
  if (!p) return MOE_OK;
  cudaSetDevice(p->device);
  cudaDeviceSynchronize();
  free_ep(p);
  return MOE_OK;
}

moe_status moe_ep_forward(moe_ep* p, const void* x, const int32_t* ids, const float* w, int T, const uint8_t* w13,
                          const uint8_t* w13s, const uint8_t* w2, const uint8_t* w2s, int act, float beta, float lbeta,
                          int adt, void* out, void* stream) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "ep is NULL");
  if (T < 0 || T > p->max_tokens) return fail(MOE_ERR_INVALID_ARG, "num_tokens %d outside [0, %d]", T, p->max_tokens);
  if (T == 0) return MOE_OK;
  const void* ptrs[] = {x, ids, w, w13, w13s, w2, w2s, out};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return fail(MOE_ERR_INVALID_ARG, "NULL or misaligned tensor pointer");
  CUDA_TRY(cudaSetDevice(p->device));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int H = p->H, I = p->I, El = p->El, R = p->R, K = p->K, M = p->max_tokens;
  // dispatch: each rank's received rows, then the counts to the host (one sync)
  cudaError_t e = launch_ep_dispatch(x, ids, w, T, H, K, El, R, M, p->recv_tok, p->recv_ids, p->recv_w, p->slot,
                                     p->counts, p->recv_x, p->rank[0]->err, p->num_sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "dispatch launch");
  CUDA_TRY(cudaMemcpyAsync(p->counts_h, p->counts, sizeof(int32_t) * R, cudaMemcpyDeviceToHost, st));
  CUDA_TRY(cudaStreamSynchronize(st));
  // each rank: its received rows against its slice of the experts, fp32 shares kept
  EpShares sh{};
  for (int r = 0; r < R; ++r) {
    const size_t e0 = (size_t)r * El;
    const uint8_t* rw13 = w13 + e0 * 2 * I * (H / 2);
    const uint8_t* rw13s = w13s + e0 * 2 * I * (H / 32);
    const uint8_t* rw2 = w2 + e0 * H * (I / 2);
    const uint8_t* rw2s = w2s + e0 * H * (I / 32);
    const int Tr = p->counts_h[r];
    sh.acc[r] = p->rank[r]->acc32;
    if (Tr == 0) continue;
    moe_status s = forward_impl(p->rank[r], static_cast<const uint8_t*>(p->recv_x) + (size_t)r * M * H * 2,
                                p->recv_ids + (size_t)r * M * K, p->recv_w + (size_t)r * M * K, Tr, rw13, rw13s, rw2,
                                rw2s, act, beta, lbeta, adt, nullptr, stream, true);
    if (s != MOE_OK) return s;
  }
  // combine: each rank's shares over the fp8 1x32 wire, summed per token
  e = launch_ep_combine(sh, p->counts, p->slot, T, H, R, M, p->wire_q, p->wire_s, out, p->num_sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return MOE_OK;
}

moe_status moe_ep_counts(moe_ep* p, int32_t* counts) {
  if (!p || !counts) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
  for (int r = 0; r < p->R; ++r) counts[r] = p->counts_h[r];
  return MOE_OK;
}

moe_status moe_ep_get_error(moe_ep* p, int32_t* flags) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "ep is NULL");
  int32_t all = 0;
  moe_status worst = MOE_OK;
  for (int r = 0; r < p->R; ++r) {
    int32_t f = 0;
    moe_status s = moe_get_error(p->rank[r], &f);
    all |= f;
    if (s != MOE_OK && worst == MOE_OK) worst = s;
  }
  if (flags) *flags = all;
  return worst;
}

moe_status moe_forward(moe_ctx* c, const void* x, const int32_t* ids, const float* w, int T, const uint8_t* w13,
                       const uint8_t* w13s, const uint8_t* w2, const uint8_t* w2s, int act, float beta,
                       float lbeta, int adt, void* out, void* stream) {
  if (T > 0 && !out) return fail(MOE_ERR_INVALID_ARG, "NULL tensor pointer");
  return forward_impl(c, x, ids, w, T, w13, w13s, w2, w2s, act, beta, lbeta, adt, out, stream, false);
}

moe_status moe_forward_host(moe_ctx* c, const void* x_host, const int32_t* ids_host, const float* w_host, int T,
                            const uint8_t* w13, const uint8_t* w13s, const uint8_t* w2, const uint8_t* w2s, int act,
                            float beta, float lbeta, int adt, void* out_host, void* stream) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "ctx is NULL");
  if (T < 0 || T > c->max_tokens) return fail(MOE_ERR_INVALID_ARG, "num_tokens %d outside [0, %d]", T, c->max_tokens);
  if (T == 0) return MOE_OK;
  if (!x_host || !ids_host || !w_host || !out_host) return fail(MOE_ERR_INVALID_ARG, "NULL host buffer");
  CUDA_TRY(cudaSetDevice(c->device));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t xb = (size_t)T * c->H * 2, pb = (size_t)T * c->K;
  // Page-locked host memory the device can address is used in place (the kernels
  // read x, ids and weights and write out across the host link: no copy launches);
  // anything else goes through the device staging buffers.
  auto in_place = [&](const void* h) -> void* {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
      cudaGetLastError();  // (clear: an unknown pointer is not an error here)
      return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
  };
  const void* x = in_place(x_host);
  const int32_t* ids = static_cast<const int32_t*>(in_place(ids_host));
  const float* w = static_cast<const float*>(in_place(w_host));
  void* out = in_place(out_host);
  if (!x) {
    CUDA_TRY(cudaMemcpyAsync(c->st_x, x_host, xb, cudaMemcpyHostToDevice, st));
    x = c->st_x;
  }
  if (!ids) {
    CUDA_TRY(cudaMemcpyAsync(c->st_ids, ids_host, pb * sizeof(int32_t), cudaMemcpyHostToDevice, st));
    ids = c->st_ids;
  }
  if (!w) {
    CUDA_TRY(cudaMemcpyAsync(c->st_w, w_host, pb * sizeof(float), cudaMemcpyHostToDevice, st));
    w = c->st_w;
  }
  moe_status s = moe_forward(c, x, ids, w, T, w13, w13s, w2, w2s, act, beta, lbeta, adt, out ? out : c->st_out,
                             stream);
  if (s != MOE_OK) {
    cudaStreamSynchronize(st);  // copies already enqueued finish before the caller reuses its buffers
    return s;
  }
  if (!out) CUDA_TRY(cudaMemcpyAsync(out_host, c->st_out, xb, cudaMemcpyDeviceToHost, st));
  CUDA_TRY(cudaStreamSynchronize(st));
  return MOE_OK;
}

moe_status moe_quantize_activations(const void* x, int T, int H, int adt, uint8_t* codes, uint8_t* scales,
                                    void* stream) {
  if (T < 0 || H <= 0 || H % 32) return fail(MOE_ERR_INVALID_ARG, "bad sizes T=%d H=%d (H %% 32 == 0)", T, H);
  if (adt != MOE_A_BF16 && adt != MOE_A_FP8 && adt != MOE_A_FP4) return fail(MOE_ERR_UNSUPPORTED, "a_dtype %d unknown", adt);
  if (T == 0) return MOE_OK;
  if (!x || !codes || !scales) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  int dev = 0, sms = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  cudaError_t e = launch_act_quant(x, T, H, fmt_of_adtype(adt), codes, scales, H / 32, nullptr, sms,
                                   reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "activation quantisation launch");
  return MOE_OK;
}

moe_status moe_route(const float* logits, int T, int E, int K, int32_t* ids, float* weights, void* stream) {
  if (T < 0 || E <= 0 || E > ROUTE_MAX_EXPERTS || K <= 0 || K > E || K > ROUTE_MAX_TOPK)
    return fail(MOE_ERR_INVALID_ARG, "bad sizes T=%d E=%d K=%d (1 <= K <= min(E, %d), E <= %d)", T, E, K,
                ROUTE_MAX_TOPK, ROUTE_MAX_EXPERTS);
  if (T == 0) return MOE_OK;
  if (!logits || !ids || !weights) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  int dev = 0, sms = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  static std::once_flag once[64];
  cudaError_t se = cudaSuccess;
  if (dev >= 0 && dev < 64) std::call_once(once[dev], [&] { se = route_set_smem_limits(); });
  if (se != cudaSuccess) return cuda_fail(se, "router kernel attributes");
  cudaError_t e = launch_route(logits, T, E, K, ids, weights, sms, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "router launch");
  return MOE_OK;
}

moe_status moe_quantize_mxfp4(const float* w, int64_t rows, int cols, uint8_t* codes, uint8_t* scales, void* stream) {
  if (rows < 0 || cols <= 0 || cols % 32) return fail(MOE_ERR_INVALID_ARG, "bad sizes rows=%lld cols=%d", (long long)rows, cols);
  if (rows == 0) return MOE_OK;
  if (!w || !codes || !scales) return fail(MOE_ERR_INVALID_ARG, "NULL pointer");
  int dev = 0, sms = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  cudaError_t e = launch_weight_quant(w, rows * (cols / 32), codes, scales, sms, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "weight quantisation launch");
  return MOE_OK;
}

moe_status moe_set_profiling(moe_ctx* c, int enable) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "ctx is NULL");
  CUDA_TRY(cudaSetDevice(c->device));
  if (enable && !c->ev[0])
    for (cudaEvent_t& e : c->ev) CUDA_TRY(cudaEventCreate(&e));
  c->profiling = enable ? 1 : 0;
  c->ev_n = 0;
  return MOE_OK;
}

moe_status moe_read_profile(moe_ctx* c, float* ms, const char** names, int* count) {
  if (!c || !count) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
  if (!c->profiling || c->ev_n < 2) { *count = 0; return MOE_OK; }
  CUDA_TRY(cudaEventSynchronize(c->ev[c->ev_n - 1]));
  int n = c->ev_n - 1 < *count ? c->ev_n - 1 : *count;
  for (int i = 0; i < n; ++i) {
    float t = 0.f;
    CUDA_TRY(cudaEventElapsedTime(&t, c->ev[i], c->ev[i + 1]));
    if (ms) ms[i] = t;
    if (names) names[i] = c->ev_name[i];
  }
  *count = n;
  return MOE_OK;
}

moe_status moe_prepack_size(moe_ctx* c, int64_t* bytes) {
  if (!c || !bytes) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
  *bytes = (int64_t)c->E * c->H * (c->I / 2) + (int64_t)c->E * c->H * (c->I / 32);
  return MOE_OK;
}

moe_status moe_prepack(moe_ctx* c, const uint8_t* w2, const uint8_t* w2s, int a_dtype, void* packed, void* stream) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "ctx is NULL");
  if (!packed) {  // unbind
    c->pk_src = nullptr;
    c->pk_codes = c->pk_scales = nullptr;
    c->tm_w2pk_key = nullptr;
    return MOE_OK;
  }
  if (!w2 || !w2s) return fail(MOE_ERR_INVALID_ARG, "NULL weight pointer");
  if (a_dtype != MOE_A_BF16 && a_dtype != MOE_A_FP8 && a_dtype != MOE_A_FP4)
    return fail(MOE_ERR_UNSUPPORTED, "a_dtype %d unknown", a_dtype);
  if (!aligned16(w2) || !aligned16(w2s) || !aligned16(packed))
    return fail(MOE_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  CUDA_TRY(cudaSetDevice(c->device));
  uint8_t* pc = static_cast<uint8_t*>(packed);
  uint8_t* ps = pc + (size_t)c->E * c->H * (c->I / 2);
  // kind::mxf4 (bf16 and fp4 activations) reads the blocks pre-swizzled by one bulk copy;
  // kind::mxf8f6f4 (fp8) through the unpacking TMA, rows in order
  cudaError_t e = launch_prepack_w2(w2, w2s, c->E, c->H, c->I, a_dtype != MOE_A_FP8, pc, ps, c->num_sms,
                                    reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "prepack launch");
  c->pk_src = w2;
  c->pk_adt = a_dtype;
  c->pk_codes = pc;
  c->pk_scales = ps;
  c->tm_w2pk_key = nullptr;
  return MOE_OK;
}

moe_status moe_debug_inject(int what, int64_t arg) {
  if (what != MOE_INJECT_ALLOC_FAIL) return fail(MOE_ERR_INVALID_ARG, "unknown injection %d", what);
  g_fail_alloc.store(arg < 0 ? -1 : (long)arg);
  return MOE_OK;
}

moe_status moe_selftest_wait(moe_ctx* c, int64_t limit_ns, int complete, void* stream) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "ctx is NULL");
  if (limit_ns < 0 || limit_ns > 10000000000LL) return fail(MOE_ERR_INVALID_ARG, "limit_ns outside [0, 1e10]");
  CUDA_TRY(cudaSetDevice(c->device));
  cudaError_t e = launch_wait_selftest((uint64_t)limit_ns, complete, c->err, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wait self-test launch");
  return MOE_OK;
}

moe_status moe_get_error(moe_ctx* c, int32_t* flags) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "ctx is NULL");
  CUDA_TRY(cudaSetDevice(c->device));
  CUDA_TRY(cudaDeviceSynchronize());
  int v = 0;
  CUDA_TRY(cudaMemcpy(&v, c->err, sizeof(int), cudaMemcpyDeviceToHost));
  CUDA_TRY(cudaMemset(c->err, 0, sizeof(int)));
  if (flags) *flags = v;
  if (v & DEV_ERR_LAUNCH) return fail(MOE_ERR_CUDA, "a kernel was launched with too little shared memory");
  if (v & DEV_ERR_TIMEOUT) return MOE_ERR_TIMEOUT;
  if (v & DEV_ERR_BAD_EXPERT) return MOE_ERR_BAD_EXPERT_ID;
  return MOE_OK;
}

}  // extern "C"
