// C ABI of libcoli_moe.so: contexts, weight upload, the expert table, error reporting and the
// argument checks of the compute calls. The kernels live in router.cu and experts.cu.
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <string>

#include "coli_internal.h"
#include "ans.h"
#include "ep.h"

namespace coli {

int fail(coli_ctx* ctx, int code, const std::string& msg) {
  if (ctx) {
    ctx->last_error = msg;
    ctx->last_code = code;
  }
  return code;
}

// Record a failed runtime call and consume the runtime's error state so that the next healthy
// call does not report it (a failed allocation must not poison later launches).
int cuda_fail(coli_ctx* ctx, cudaError_t e, const char* what) {
  (void)cudaGetLastError();
  std::string m = std::string(what) + ": " + cudaGetErrorString(e);
  return fail(ctx, e == cudaErrorMemoryAllocation ? COLI_E_OOM : COLI_E_CUDA, m);
}

bool injected(coli_ctx* ctx) {
  if (ctx->fail_after < 0) return false;
  if (ctx->compute_calls >= ctx->fail_after) {
    ctx->last_error = "COLI_FAIL_AFTER test hook";
    ctx->last_code = COLI_E_INJECTED;
    return true;
  }
  return false;
}

int ensure_workspace(coli_ctx* ctx, size_t bytes) {
  bytes = align_up(bytes < 256 ? 256 : bytes, 256);
  if (bytes <= ctx->ws.bytes) return COLI_OK;
  if (ctx->ws.base) {
    cudaError_t e = cudaStreamSynchronize(ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "workspace grow: stream sync");
    cudaFree(ctx->ws.base);
    ctx->ws.base = nullptr;
    ctx->ws.bytes = 0;
  }
  void* p = nullptr;
  cudaError_t e = cudaMalloc(&p, bytes);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "workspace cudaMalloc");
  ctx->ws.base = static_cast<char*>(p);
  ctx->ws.bytes = bytes;
  return COLI_OK;
}

// The issue/take slot pool. It only grows at the first issue of a round (or in coli_reserve), when no
// slot holds a pending partial sum; the old pool is freed after the stream has drained.
int ensure_slots(coli_ctx* ctx, size_t bytes) {
  bytes = align_up(bytes < 256 ? 256 : bytes, 256);
  if (bytes <= ctx->slot_bytes) return COLI_OK;
  if (ctx->slots) {
    cudaError_t e = cudaStreamSynchronize(ctx->stream);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "slot pool grow: stream sync");
    cudaFree(ctx->slots);
    ctx->slots = nullptr;
    ctx->slot_bytes = 0;
  }
  void* p = nullptr;
  cudaError_t e = cudaMalloc(&p, bytes);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "slot pool cudaMalloc");
  ctx->slots = static_cast<float*>(p);
  ctx->slot_bytes = bytes;
  return COLI_OK;
}

static cudaEvent_t prof_event(coli_ctx* ctx) {
  if (!ctx->prof_free.empty()) {
    cudaEvent_t e = ctx->prof_free.back();
    ctx->prof_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return e;
}

ProfScope::ProfScope(coli_ctx* c, int k) : ctx(c), kind(k) {
  if (!ctx->prof) return;
  a = prof_event(ctx);
  b = prof_event(ctx);
  if (a) cudaEventRecord(a, ctx->stream);
}

ProfScope::~ProfScope() {
  if (!ctx->prof) return;
  if (a && b && cudaEventRecord(b, ctx->stream) == cudaSuccess) {
    ctx->prof_pending.push_back({kind, a, b});
  } else {
    (void)cudaGetLastError();
    if (a) ctx->prof_free.push_back(a);
    if (b) ctx->prof_free.push_back(b);
  }
}

static bool valid_handle(coli_ctx* ctx, uint64_t h) {
  return h >= 1 && h <= ctx->tensors.size() && ctx->tensors[h - 1].live;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link-time libcuda dependency).
static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    (void)cudaGetLastError();
  }
  return fn;
}

// Device descriptor of an uploaded tensor, with its TMA maps: the weights as a uint32 matrix
// [O x pitch/4] read in boxes of [min(kBoxRows, O) rows x one warp's 128-word column slice], and,
// when the group size lets a warp's chunk-group scales form a 16-byte-multiple box, the scales.
static int make_desc(coli_ctx* ctx, HostTensor& t) {
  TensorDesc d{};
  d.w = t.w;
  d.s = t.s;
  d.pitch = t.pitch;
  d.gs = t.gs;
  d.G = t.G;
  d.rows = t.O;
  d.cols = t.I;
  d.mode = t.gs == 0 ? SCALE_ROW : (t.gs % 32 == 0 ? SCALE_CHUNK : SCALE_GENERIC);
  const uint32_t words = t.pitch / 4;
  d.box_rows = t.O < kBoxRows ? (uint32_t)t.O : (uint32_t)kBoxRows;
  d.box_w = words < (uint32_t)kSliceWords ? words : (uint32_t)kSliceWords;
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(ctx, COLI_E_CUDA, "upload: cuTensorMapEncodeTiled unavailable");
  {
    cuuint64_t dims[2] = {words, (cuuint64_t)t.O};
    cuuint64_t strides[1] = {t.pitch};
    cuuint32_t box[2] = {d.box_w, d.box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(&d.map_w, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, t.w, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ctx, COLI_E_CUDA, "upload: weight tensor map encoding failed");
  }
  {
    cuuint64_t dims[2] = {words, (cuuint64_t)t.O};
    cuuint64_t strides[1] = {t.pitch};
    cuuint32_t box[2] = {(cuuint32_t)kTcWords, (cuuint32_t)kTcRows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(&d.map_tc, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, t.w, dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ctx, COLI_E_CUDA, "upload: tensor-core tile map encoding failed");
  }
  d.box_s = 0;
  if (d.mode == SCALE_CHUNK && t.gs >= 64 && t.gs <= 256 && t.G % 4 == 0) {
    uint32_t per_warp = (uint32_t)(32 * 32 / t.gs);  // chunk groups under one warp's 32 chunks
    uint32_t bs = per_warp < (uint32_t)t.G ? per_warp : (uint32_t)t.G;
    cuuint64_t dims[2] = {(cuuint64_t)t.G, (cuuint64_t)t.O};
    cuuint64_t strides[1] = {(cuuint64_t)t.G * 4};
    cuuint32_t box[2] = {bs, d.box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(&d.map_s, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, t.s, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS) d.box_s = bs;
  }
  t.desc = d;
  return COLI_OK;
}

int encode_bf16_rows_map(coli_ctx* ctx, CUtensorMap* map, void* base, long long rows, int cols) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(ctx, COLI_E_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, 16};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ctx, COLI_E_CUDA, "activation tensor map encoding failed");
  return COLI_OK;
}

}  // namespace coli

using namespace coli;

extern "C" {

int coli_init(coli_ctx** out, int device, void* cuda_stream) {
  if (!out) return COLI_E_INVAL;
  *out = nullptr;
  int n = 0;
  cudaError_t e = cudaGetDeviceCount(&n);
  if (e != cudaSuccess || device < 0 || device >= n) {
    (void)cudaGetLastError();
    return COLI_E_CUDA;
  }
  if ((e = cudaSetDevice(device)) != cudaSuccess) {
    (void)cudaGetLastError();
    return COLI_E_CUDA;
  }
  coli_ctx* ctx = new coli_ctx();
  ctx->device = device;
  ctx->stream = static_cast<cudaStream_t>(cuda_stream);
  cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, device);
  const char* fa = getenv("COLI_FAIL_AFTER");
  if (fa && *fa) ctx->fail_after = atoll(fa);
  const char* fu = getenv("COLI_DECODE_FUSED");
  if (fu && *fu) ctx->decode_fused = atoi(fu) != 0;
  const char* fs = getenv("COLI_DECODE_STREAM");
  if (fs && *fs) ctx->stream_ffn = atoi(fs) != 0;
  const char* tw = getenv("COLI_TEST_WAIT_NS");
  if (tw && *tw) ctx->wait_ns = strtoull(tw, nullptr, 10);
  const char* th = getenv("COLI_TEST_WITHHOLD");
  if (th && *th) ctx->test_withhold = atoi(th) != 0;
  const char* thr = getenv("COLI_TEST_WITHHOLD_ROUTER");
  if (thr && *thr) ctx->test_withhold_router = atoi(thr);
  const char* rr = getenv("COLI_ROUTER_ROWS");
  if (rr && *rr) ctx->router_rows = atoi(rr);
  if (ctx->router_rows != 1 && ctx->router_rows != 2 && ctx->router_rows != 4 && ctx->router_rows != 8)
    ctx->router_rows = 0;
  const char* rp = getenv("COLI_ROUTER_PARTS");
  if (rp && *rp) ctx->router_parts = std::max(0, std::min(4, atoi(rp)));
  ctx->h_table.assign(COLI_MAX_EXPERTS, ExpertDesc{});
  ctx->table_handles.assign(3 * COLI_MAX_EXPERTS, 0);
  ctx->table_stream.assign(COLI_MAX_EXPERTS, 1);
  void* p = nullptr;
  if ((e = cudaMalloc(&p, sizeof(ExpertDesc) * COLI_MAX_EXPERTS)) != cudaSuccess) goto fail;
  ctx->d_table = static_cast<ExpertDesc*>(p);
  if ((e = cudaMemset(ctx->d_table, 0, sizeof(ExpertDesc) * COLI_MAX_EXPERTS)) != cudaSuccess) goto fail;
  if ((e = cudaMalloc(&p, kStatusBytes)) != cudaSuccess) goto fail;
  ctx->d_status = static_cast<int*>(p);
  if ((e = cudaMemset(ctx->d_status, 0, kStatusBytes)) != cudaSuccess) goto fail;
  if ((e = cudaMalloc(&ctx->d_router, kRouterScratchBytes)) != cudaSuccess) goto fail;
  if ((e = cudaMemset(ctx->d_router, 0, kRouterScratchBytes)) != cudaSuccess) goto fail;
  {
    const int32_t route[2] = {0, 0x3f800000};  // expert 0, then the bits of 1.0f
    if ((e = cudaMalloc(&p, sizeof(route))) != cudaSuccess) goto fail;
    ctx->d_solo_route = static_cast<int32_t*>(p);
    if ((e = cudaMemcpy(ctx->d_solo_route, route, sizeof(route), cudaMemcpyHostToDevice)) != cudaSuccess) goto fail;
  }
  ctx->coop_mode = probe_coop_mode(ctx);
  *out = ctx;
  return COLI_OK;
fail:
  (void)cudaGetLastError();
  coli_destroy(ctx);
  return e == cudaErrorMemoryAllocation ? COLI_E_OOM : COLI_E_CUDA;
}

void coli_destroy(coli_ctx* ctx) {
  if (!ctx) return;
  cudaSetDevice(ctx->device);
  cudaStreamSynchronize(ctx->stream);
  for (auto& t : ctx->tensors) {
    if (t.w) cudaFree(t.w);
    if (t.s) cudaFree(t.s);
    if (t.d_solo) cudaFree(t.d_solo);
    if (t.panel) cudaFree(t.panel);
    if (t.sT) cudaFree(t.sT);
  }
  if (ctx->d_solo_route) cudaFree(ctx->d_solo_route);
  ans_release_all(ctx);
  if (ctx->d_table) cudaFree(ctx->d_table);
  if (ctx->d_status) cudaFree(ctx->d_status);
  if (ctx->d_router) cudaFree(ctx->d_router);
  if (ctx->ws.base) cudaFree(ctx->ws.base);
  if (ctx->slots) cudaFree(ctx->slots);
  for (auto& r : ctx->prof_pending) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto ev : ctx->prof_free) cudaEventDestroy(ev);
  (void)cudaGetLastError();
  delete ctx;
}

int coli_set_stream(coli_ctx* ctx, void* cuda_stream) {
  if (!ctx) return COLI_E_INVAL;
  ctx->stream = static_cast<cudaStream_t>(cuda_stream);
  return COLI_OK;
}

const char* coli_last_error(coli_ctx* ctx) { return ctx ? ctx->last_error.c_str() : "null context"; }

int coli_last_code(coli_ctx* ctx) { return ctx ? ctx->last_code : COLI_E_INVAL; }

int coli_check_error(coli_ctx* ctx) {
  if (!ctx) return COLI_E_INVAL;
  cudaSetDevice(ctx->device);
  cudaError_t e = cudaStreamSynchronize(ctx->stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "coli_check_error: stream sync");
  int code = 0;
  e = cudaMemcpy(&code, ctx->d_status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "coli_check_error: read error word");
  if (code != 0) {
    // after a timed-out wait the synchronisation words may be left mid-count: clear them with the
    // error word
    e = cudaMemset(ctx->d_status, 0, code == COLI_E_TIMEOUT ? kStatusBytes : sizeof(int));
    if (e != cudaSuccess) return cuda_fail(ctx, e, "coli_check_error: clear error word");
    ctx->last_error = code == COLI_E_ROUTE ? "device: expert index out of range or unset table entry"
                      : code == COLI_E_NONFINITE ? "device: non-finite activation or router score"
                      : code == COLI_E_TIMEOUT   ? "device: a bounded wait inside a kernel gave up"
                                                 : "device error";
  }
  return code;
}

int coli_profile_enable(coli_ctx* ctx, int on) {
  if (!ctx) return COLI_E_INVAL;
  ctx->prof = on != 0;
  return COLI_OK;
}

int coli_profile_read(coli_ctx* ctx, int kind, double* total_ms, long long* launches) {
  if (!ctx || kind < 0 || kind > COLI_KERNEL_LINEAR || !total_ms || !launches) return COLI_E_INVAL;
  cudaSetDevice(ctx->device);
  cudaError_t e = cudaStreamSynchronize(ctx->stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "coli_profile_read: stream sync");
  for (auto& r : ctx->prof_pending) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
      ctx->prof_ms[r.kind] += ms;
      ctx->prof_n[r.kind] += 1;
    } else {
      (void)cudaGetLastError();
    }
    ctx->prof_free.push_back(r.a);
    ctx->prof_free.push_back(r.b);
  }
  ctx->prof_pending.clear();
  *total_ms = ctx->prof_ms[kind];
  *launches = ctx->prof_n[kind];
  ctx->prof_ms[kind] = 0;
  ctx->prof_n[kind] = 0;
  return COLI_OK;
}

int coli_reserve(coli_ctx* ctx, int max_S, int max_E, int max_K, int max_D, int max_I) {
  if (!ctx || max_S < 1 || max_E < 1 || max_K < 1 || max_D < 1 || max_I < 1) return COLI_E_INVAL;
  size_t router = align_up((size_t)max_S * max_E * 2 * sizeof(float), 256);
  const size_t routes = (size_t)max_S * max_K;
  // grouped GEMV path: h, per-route rows (S > 1) or the fused kernel's partial rows (S == 1), plan
  size_t experts = align_up(routes * max_I * sizeof(float), 256) +
                   align_up((routes > (size_t)max_K * kFusedMaxSlices ? routes : (size_t)max_K * kFusedMaxSlices) *
                                max_D * sizeof(float), 256) +
                   4096 + align_up((size_t)(max_S + 1) * sizeof(int) * 4, 256);
  // tensor-core path: grouped rows (each expert's block padded to 16) as bf16 x and h, f32 outputs
  const size_t pf_rows = routes + 16 * (size_t)(max_E < COLI_MAX_EXPERTS ? max_E : COLI_MAX_EXPERTS) + 16;
  const size_t prefill = pf_rows * ((size_t)max_D * 2 + (size_t)max_I * 2 + (size_t)max_D * 4 + 4) + routes * 4 +
                         (size_t)max_E * 8 + (routes / 128 + max_E + 1) * 16 + 16 * 256;
  if (prefill > experts) experts = prefill;
  // one-launch S == 1 FFN: a partial row of y per CTA
  const size_t stream = (size_t)ctx->num_sms * max_D * sizeof(float);
  if (stream > experts) experts = stream;
  const size_t slots = (size_t)COLI_MAX_ISSUES * max_S * max_D * sizeof(float);
  cudaSetDevice(ctx->device);
  int rc = ensure_slots(ctx, slots);
  if (rc != COLI_OK) return rc;
  return ensure_workspace(ctx, router > experts ? router : experts);
}

uint64_t coli_expert_upload(coli_ctx* ctx, const uint8_t* packed, const float* scales, int O, int I,
                            int gs) {
  if (!ctx) return 0;
  if (!packed || !scales || O < 1 || I < 2 || O > COLI_MAX_DIM || I > COLI_MAX_DIM) {
    fail(ctx, COLI_E_INVAL, "upload: NULL pointer or shape out of range");
    return 0;
  }
  if (I % 2 != 0 || gs < 0 || gs % 2 != 0) {
    fail(ctx, COLI_E_FORMAT, "upload: I must be even and gs must be 0 or a positive even number");
    return 0;
  }
  cudaSetDevice(ctx->device);
  HostTensor t;
  t.O = O;
  t.I = I;
  t.gs = gs;
  t.G = gs == 0 ? 1 : (I + gs - 1) / gs;
  t.pitch = (uint32_t)(((I + 31) / 32) * 16);
  size_t nscales = gs == 0 ? (size_t)O : (size_t)O * t.G;
  size_t row_bytes = (size_t)I / 2;
  void* pw = nullptr;
  void* ps = nullptr;
  cudaError_t e;
  if ((e = cudaMalloc(&pw, (size_t)O * t.pitch)) != cudaSuccess) {
    cuda_fail(ctx, e, "upload: cudaMalloc weights");
    return 0;
  }
  if ((e = cudaMalloc(&ps, nscales * sizeof(float))) != cudaSuccess) {
    cudaFree(pw);
    cuda_fail(ctx, e, "upload: cudaMalloc scales");
    return 0;
  }
  // pad nibbles hold 8 (the value 0); then copy the caller's rows into the padded pitch
  if ((e = cudaMemsetAsync(pw, 0x88, (size_t)O * t.pitch, ctx->stream)) != cudaSuccess ||
      (e = cudaMemcpy2DAsync(pw, t.pitch, packed, row_bytes, row_bytes, O, cudaMemcpyDefault,
                             ctx->stream)) != cudaSuccess ||
      (e = cudaMemcpyAsync(ps, scales, nscales * sizeof(float), cudaMemcpyDefault, ctx->stream)) !=
          cudaSuccess ||
      (e = cudaStreamSynchronize(ctx->stream)) != cudaSuccess) {
    cudaFree(pw);
    cudaFree(ps);
    cuda_fail(ctx, e, "upload: copy");
    return 0;
  }
  t.w = static_cast<uint8_t*>(pw);
  t.s = static_cast<float*>(ps);
  if (make_desc(ctx, t) != COLI_OK) {
    cudaFree(pw);
    cudaFree(ps);
    return 0;
  }
  {  // a one-entry expert table whose down tensor is this one (coli_w4_linear for one token)
    ExpertDesc solo{};
    solo.t[T_DOWN] = t.desc;
    solo.valid = 1;
    void* pd = nullptr;
    if ((e = cudaMalloc(&pd, sizeof(ExpertDesc))) != cudaSuccess ||
        (e = cudaMemcpy(pd, &solo, sizeof(ExpertDesc), cudaMemcpyHostToDevice)) != cudaSuccess) {
      if (pd) cudaFree(pd);
      cudaFree(pw);
      cudaFree(ps);
      cuda_fail(ctx, e, "upload: device descriptor");
      return 0;
    }
    t.d_solo = static_cast<ExpertDesc*>(pd);
  }
  t.live = true;
  ctx->tensors.push_back(t);
  return (uint64_t)ctx->tensors.size();
}

int coli_tensor_shape(coli_ctx* ctx, uint64_t handle, int* O, int* I, int* gs) {
  if (!ctx) return COLI_E_INVAL;
  if (!valid_handle(ctx, handle)) return fail(ctx, COLI_E_INVAL, "tensor_shape: unknown tensor handle");
  const HostTensor& t = ctx->tensors[handle - 1];
  if (O) *O = t.O;
  if (I) *I = t.I;
  if (gs) *gs = t.gs;
  return COLI_OK;
}

int coli_expert_free(coli_ctx* ctx, uint64_t handle) {
  if (!ctx) return COLI_E_INVAL;
  if (!valid_handle(ctx, handle)) return fail(ctx, COLI_E_INVAL, "free: unknown handle");
  HostTensor& t = ctx->tensors[handle - 1];
  if (t.table_refs > 0) return fail(ctx, COLI_E_INVAL, "free: tensor is still in the expert table");
  cudaSetDevice(ctx->device);
  cudaError_t e = cudaStreamSynchronize(ctx->stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "free: stream sync");
  cudaFree(t.w);
  cudaFree(t.s);
  if (t.d_solo) cudaFree(t.d_solo);
  if (t.panel) cudaFree(t.panel);
  if (t.sT) cudaFree(t.sT);
  t = HostTensor{};
  return COLI_OK;
}

int coli_expert_table_set(coli_ctx* ctx, int e, uint64_t gate, uint64_t up, uint64_t down) {
  if (!ctx) return COLI_E_INVAL;
  if (e < 0 || e >= COLI_MAX_EXPERTS) return fail(ctx, COLI_E_INVAL, "table_set: expert id out of range");
  cudaSetDevice(ctx->device);
  uint64_t* cur = &ctx->table_handles[3 * (size_t)e];
  ExpertDesc d{};
  if (gate == 0 && up == 0 && down == 0) {
    if (cur[0]) {
      for (int i = 0; i < 3; i++) ctx->tensors[cur[i] - 1].table_refs--;
      if (!ctx->table_stream[e]) ctx->table_nostream--;
      ctx->table_stream[e] = 1;
      ctx->table_count--;
      if (ctx->table_count == 0) ctx->table_D = ctx->table_I = 0;
    }
    for (int i = 0; i < 3; i++) cur[i] = 0;
  } else {
    if (!valid_handle(ctx, gate) || !valid_handle(ctx, up) || !valid_handle(ctx, down))
      return fail(ctx, COLI_E_INVAL, "table_set: unknown handle");
    const HostTensor &g = ctx->tensors[gate - 1], &u = ctx->tensors[up - 1], &dn = ctx->tensors[down - 1];
    int I = g.O, D = g.I;
    if (u.O != I || u.I != D || dn.O != D || dn.I != I)
      return fail(ctx, COLI_E_FORMAT, "table_set: need gate [I x D], up [I x D], down [D x I]");
    bool replacing = cur[0] != 0;
    if (ctx->table_count - (replacing ? 1 : 0) > 0 && (ctx->table_D != D || ctx->table_I != I))
      return fail(ctx, COLI_E_FORMAT, "table_set: every expert must share D and I");
    // the one-launch S == 1 FFN streams down tensors panel-major: build that view once per tensor
    HostTensor& dnt = ctx->tensors[down - 1];
    const bool streamable = ctx->stream_ffn && stream_tensor_ok(g, false) && stream_tensor_ok(u, false) &&
                            stream_tensor_ok(dnt, true);
    if (streamable) {
      int rc = build_stream_view(ctx, dnt);
      if (rc != COLI_OK) return rc;
      const int gG = g.gs > 0 ? g.G : 0, uG = u.gs > 0 ? u.G : 0;
      ctx->table_gu_maxG = std::max(ctx->table_gu_maxG, std::max(gG, uG));
    }
    if (replacing) {
      for (int i = 0; i < 3; i++) ctx->tensors[cur[i] - 1].table_refs--;
      if (!ctx->table_stream[e]) ctx->table_nostream--;
    } else {
      ctx->table_count++;
    }
    ctx->table_stream[e] = streamable;
    if (!streamable) ctx->table_nostream++;
    ctx->table_D = D;
    ctx->table_I = I;
    cur[0] = gate;
    cur[1] = up;
    cur[2] = down;
    for (int i = 0; i < 3; i++) ctx->tensors[cur[i] - 1].table_refs++;
    d.t[T_GATE] = g.desc;
    d.t[T_UP] = u.desc;
    d.t[T_DOWN] = dnt.desc;
    d.valid = 1;
  }
  ctx->h_table[e] = d;
  cudaError_t ce = cudaMemcpyAsync(ctx->d_table + e, &ctx->h_table[e], sizeof(ExpertDesc),
                                   cudaMemcpyHostToDevice, ctx->stream);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(ctx->stream);
  if (ce != cudaSuccess) return cuda_fail(ctx, ce, "table_set: copy descriptor");
  return COLI_OK;
}

int coli_router_select(coli_ctx* ctx, const void* x, int x_dtype, int S, int D, const float* Wr,
                       const float* bias, int E, int K, float topp, int norm_topk, float routed_scale,
                       int32_t* idx, float* w, int32_t* n_sel) {
  if (!ctx) return COLI_E_INVAL;
  if (!x || !Wr || !idx || !w) return fail(ctx, COLI_E_INVAL, "router: NULL pointer");
  if (x_dtype != COLI_DTYPE_F32 && x_dtype != COLI_DTYPE_BF16) return fail(ctx, COLI_E_INVAL, "router: dtype");
  if (S < 1 || S > COLI_MAX_TOKENS || D < 1 || D > COLI_MAX_DIM || E < 1 || E > COLI_MAX_EXPERTS || K < 1 ||
      K > COLI_MAX_K || K > E)
    return fail(ctx, COLI_E_INVAL, "router: size out of range");
  if (injected(ctx)) return COLI_E_INJECTED;
  cudaSetDevice(ctx->device);
  int rc = launch_router(ctx, x, x_dtype, S, D, Wr, bias, E, K, topp, norm_topk, routed_scale, -1, idx, w, n_sel);
  if (rc == COLI_OK) ctx->compute_calls++;
  return rc;
}

int coli_router_select_shared(coli_ctx* ctx, const void* x, int x_dtype, int S, int D, const float* Wr,
                              const float* bias, int E, int K, float topp, int norm_topk, float routed_scale,
                              int shared, int32_t* idx, float* w, int32_t* n_sel) {
  if (!ctx) return COLI_E_INVAL;
  if (!x || !Wr || !idx || !w) return fail(ctx, COLI_E_INVAL, "router_shared: NULL pointer");
  if (x_dtype != COLI_DTYPE_F32 && x_dtype != COLI_DTYPE_BF16) return fail(ctx, COLI_E_INVAL, "router_shared: dtype");
  if (S < 1 || S > COLI_MAX_TOKENS || D < 1 || D > COLI_MAX_DIM || E < 1 || E > COLI_MAX_EXPERTS || K < 1 ||
      K + 1 > COLI_MAX_K || K > E || shared < 0 || shared >= COLI_MAX_EXPERTS)
    return fail(ctx, COLI_E_INVAL, "router_shared: size or shared id out of range");
  if (injected(ctx)) return COLI_E_INJECTED;
  cudaSetDevice(ctx->device);
  int rc = launch_router(ctx, x, x_dtype, S, D, Wr, bias, E, K, topp, norm_topk, routed_scale, shared, idx, w, n_sel);
  if (rc == COLI_OK) ctx->compute_calls++;
  return rc;
}

int coli_router_select_noalloc(coli_ctx* ctx, const void* x, int x_dtype, int S, int D, const float* Wr,
                               const float* bias, int E, int K, float topp, int norm_topk, float routed_scale,
                               int32_t* idx, float* w, int32_t* n_sel) {
  if (!ctx) return COLI_E_INVAL;
  if (!x || !Wr || !idx || !w) return fail(ctx, COLI_E_INVAL, "router_noalloc: NULL pointer");
  if (x_dtype != COLI_DTYPE_F32 && x_dtype != COLI_DTYPE_BF16) return fail(ctx, COLI_E_INVAL, "router_noalloc: dtype");
  if (S < 1 || S > COLI_MAX_TOKENS || D < 1 || D > COLI_MAX_DIM || E < 1 || E > COLI_MAX_EXPERTS || K < 1 ||
      K > COLI_MAX_K || K > E)
    return fail(ctx, COLI_E_INVAL, "router_noalloc: size out of range");
  if (injected(ctx)) return COLI_E_INJECTED;
  cudaSetDevice(ctx->device);
  int rc = launch_router_noalloc(ctx, x, x_dtype, S, D, Wr, bias, E, K, topp, norm_topk, routed_scale, -1, idx, w,
                                  n_sel);
  if (rc == COLI_OK) ctx->compute_calls++;
  return rc;
}

int coli_expert_group(coli_ctx* ctx, const void* x_rows, int x_dtype, int S, const int32_t* idx,
                      const float* w, const int32_t* n_sel, int K, const void* resid, void* y) {
  if (!ctx) return COLI_E_INVAL;
  if (!x_rows || !idx || !w || !y) return fail(ctx, COLI_E_INVAL, "expert_group: NULL pointer");
  if (x_dtype != COLI_DTYPE_F32 && x_dtype != COLI_DTYPE_BF16)
    return fail(ctx, COLI_E_INVAL, "expert_group: dtype");
  if (S < 1 || S > COLI_MAX_TOKENS || K < 1 || K > COLI_MAX_K)
    return fail(ctx, COLI_E_INVAL, "expert_group: size out of range");
  if (ctx->table_count == 0) return fail(ctx, COLI_E_INVAL, "expert_group: expert table is empty");
  if (injected(ctx)) return COLI_E_INJECTED;
  cudaSetDevice(ctx->device);
  int rc = launch_expert_group(ctx, x_rows, x_dtype, S, idx, w, n_sel, K, resid, y, x_dtype);
  if (rc == COLI_OK) ctx->compute_calls++;
  return rc;
}

int coli_w4_linear(coli_ctx* ctx, uint64_t W, const void* x, int x_dtype, int S, const void* resid, void* y) {
  if (!ctx) return COLI_E_INVAL;
  if (!x || !y) return fail(ctx, COLI_E_INVAL, "w4_linear: NULL pointer");
  if (x_dtype != COLI_DTYPE_F32 && x_dtype != COLI_DTYPE_BF16) return fail(ctx, COLI_E_INVAL, "w4_linear: dtype");
  if (S < 1 || S > COLI_MAX_TOKENS) return fail(ctx, COLI_E_INVAL, "w4_linear: S out of range");
  if (!valid_handle(ctx, W)) return fail(ctx, COLI_E_INVAL, "w4_linear: unknown tensor handle");
  if (injected(ctx)) return COLI_E_INJECTED;
  cudaSetDevice(ctx->device);
  const HostTensor& t = ctx->tensors[W - 1];
  // one token through a tensor whose rows and scales can be streamed in 16-row units: the streaming kernel
  int rc = S == 1 && ctx->stream_ffn && stream_linear_ok(t) ? launch_stream_linear(ctx, t, x, x_dtype, resid, y)
                                                           : launch_linear(ctx, t.desc, t.d_solo, x, x_dtype, S, resid, y);
  if (rc == COLI_OK) ctx->compute_calls++;
  return rc;
}

int coli_ans_encode_host(const uint8_t* bytes, uint64_t n, uint8_t* out, uint64_t cap, uint64_t* out_len) {
  if (!bytes || n < 1 || !out_len) return COLI_E_INVAL;
  std::vector<uint8_t> blob;
  ans_encode(bytes, n, blob);
  *out_len = blob.size();
  if (!out || cap < blob.size()) return COLI_E_INVAL;
  memcpy(out, blob.data(), blob.size());
  return COLI_OK;
}

uint64_t coli_ans_upload(coli_ctx* ctx, const uint8_t* bytes, uint64_t n) {
  if (!ctx) return 0;
  if (!bytes || n < 1) {
    fail(ctx, COLI_E_INVAL, "ans_upload: NULL pointer or empty stream");
    return 0;
  }
  std::vector<uint8_t> blob;
  ans_encode(bytes, n, blob);
  cudaSetDevice(ctx->device);
  void* p = nullptr;
  cudaError_t e;
  if ((e = cudaMalloc(&p, blob.size())) != cudaSuccess) {
    cuda_fail(ctx, e, "ans_upload: cudaMalloc");
    return 0;
  }
  if ((e = cudaMemcpy(p, blob.data(), blob.size(), cudaMemcpyHostToDevice)) != cudaSuccess) {
    cudaFree(p);
    cuda_fail(ctx, e, "ans_upload: copy");
    return 0;
  }
  AnsStream st;
  st.d_blob = static_cast<uint8_t*>(p);
  st.stored = blob.size();
  st.raw = n;
  st.blocks = ans_blocks(blob.data());
  auto& v = ans_streams(ctx);
  v.push_back(st);
  return (uint64_t)v.size();
}

static AnsStream* ans_stream(coli_ctx* ctx, uint64_t h) {
  auto& v = ans_streams(ctx);
  return (h >= 1 && h <= v.size() && v[h - 1].d_blob) ? &v[h - 1] : nullptr;
}

int coli_ans_info(coli_ctx* ctx, uint64_t h, uint64_t* raw_bytes, uint64_t* stored_bytes) {
  if (!ctx) return COLI_E_INVAL;
  AnsStream* st = ans_stream(ctx, h);
  if (!st) return fail(ctx, COLI_E_INVAL, "ans_info: unknown handle");
  if (raw_bytes) *raw_bytes = st->raw;
  if (stored_bytes) *stored_bytes = st->stored;
  return COLI_OK;
}

int coli_ans_decode(coli_ctx* ctx, uint64_t h, uint8_t* out) {
  if (!ctx) return COLI_E_INVAL;
  AnsStream* st = ans_stream(ctx, h);
  if (!st) return fail(ctx, COLI_E_INVAL, "ans_decode: unknown handle");
  if (!out) return fail(ctx, COLI_E_INVAL, "ans_decode: NULL pointer");
  if (injected(ctx)) return COLI_E_INJECTED;
  cudaSetDevice(ctx->device);
  int rc = launch_ans_decode(ctx, st->d_blob, st->blocks, out);
  if (rc == COLI_OK) ctx->compute_calls++;
  return rc;
}

int coli_ans_w4_linear(coli_ctx* ctx, uint64_t h, const float* scales, int O, int I, int gs, const void* x,
                       int x_dtype, const void* resid, void* y) {
  if (!ctx) return COLI_E_INVAL;
  AnsStream* st = ans_stream(ctx, h);
  if (!st) return fail(ctx, COLI_E_INVAL, "ans_w4_linear: unknown handle");
  if (!scales || !x || !y) return fail(ctx, COLI_E_INVAL, "ans_w4_linear: NULL pointer");
  if (x_dtype != COLI_DTYPE_F32 && x_dtype != COLI_DTYPE_BF16) return fail(ctx, COLI_E_INVAL, "ans_w4_linear: dtype");
  if (O < 1 || I < 256 || I > 16384 || I % 2 || gs < 0 || gs % 2 || (uint64_t)O * (uint64_t)(I / 2) != st->raw)
    return fail(ctx, COLI_E_INVAL, "ans_w4_linear: shape does not match the stream (O rows of I/2 bytes, I even, 256 <= I <= 16384)");
  if (injected(ctx)) return COLI_E_INJECTED;
  cudaSetDevice(ctx->device);
  int rc = launch_ans_gemv(ctx, *st, scales, O, I, gs, x, x_dtype, resid, y);
  if (rc == COLI_OK) ctx->compute_calls++;
  return rc;
}

int coli_ans_free(coli_ctx* ctx, uint64_t h) {
  if (!ctx) return COLI_E_INVAL;
  AnsStream* st = ans_stream(ctx, h);
  if (!st) return fail(ctx, COLI_E_INVAL, "ans_free: unknown handle");
  cudaSetDevice(ctx->device);
  cudaError_t e = cudaStreamSynchronize(ctx->stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "ans_free: stream sync");
  cudaFree(st->d_blob);
  *st = AnsStream{};
  return COLI_OK;
}

int coli_routes_shard(coli_ctx* ctx, const int32_t* idx, const float* w, const int32_t* n_sel, int S, int K, int rank,
                      int world, int32_t* idx_out, float* w_out, int32_t* n_out) {
  if (!ctx) return COLI_E_INVAL;
  if (!idx || !w || !idx_out || !w_out || !n_out) return fail(ctx, COLI_E_INVAL, "routes_shard: NULL pointer");
  if (S < 1 || S > COLI_MAX_TOKENS || K < 1 || K > COLI_MAX_K || world < 1 || rank < 0 || rank >= world)
    return fail(ctx, COLI_E_INVAL, "routes_shard: size, rank or world out of range");
  if (injected(ctx)) return COLI_E_INJECTED;
  cudaSetDevice(ctx->device);
  int rc = launch_routes_shard(ctx, idx, w, n_sel, S, K, rank, world, idx_out, w_out, n_out);
  if (rc == COLI_OK) ctx->compute_calls++;
  return rc;
}

int coli_partials_reduce(coli_ctx* ctx, const float* parts, int n, int S, int D, const void* resid, int dtype,
                         void* y) {
  if (!ctx) return COLI_E_INVAL;
  if (!parts || !y) return fail(ctx, COLI_E_INVAL, "partials_reduce: NULL pointer");
  if (dtype != COLI_DTYPE_F32 && dtype != COLI_DTYPE_BF16) return fail(ctx, COLI_E_INVAL, "partials_reduce: dtype");
  if (n < 1 || S < 1 || S > COLI_MAX_TOKENS || D < 1 || D > COLI_MAX_DIM)
    return fail(ctx, COLI_E_INVAL, "partials_reduce: size out of range");
  if (injected(ctx)) return COLI_E_INJECTED;
  cudaSetDevice(ctx->device);
  int rc = launch_partials_reduce(ctx, parts, n, S, D, resid, dtype, y);
  if (rc == COLI_OK) ctx->compute_calls++;
  return rc;
}

int coli_expert_group_issue(coli_ctx* ctx, const void* x_rows, int x_dtype, int S, const int32_t* idx,
                            const float* w, const int32_t* n_sel, int K) {
  if (!ctx) return COLI_E_INVAL;
  if (!x_rows || !idx || !w) return fail(ctx, COLI_E_INVAL, "issue: NULL pointer");
  if (x_dtype != COLI_DTYPE_F32 && x_dtype != COLI_DTYPE_BF16) return fail(ctx, COLI_E_INVAL, "issue: dtype");
  if (S < 1 || S > COLI_MAX_TOKENS || K < 1 || K > COLI_MAX_K) return fail(ctx, COLI_E_INVAL, "issue: size out of range");
  if (ctx->table_count == 0) return fail(ctx, COLI_E_INVAL, "issue: expert table is empty");
  if (ctx->n_issued >= COLI_MAX_ISSUES) return fail(ctx, COLI_E_INVAL, "issue: COLI_MAX_ISSUES issues already pending");
  if (ctx->n_issued > 0 && (S != ctx->round_S || x_dtype != ctx->round_dtype || ctx->table_D != ctx->round_D))
    return fail(ctx, COLI_E_INVAL, "issue: S, dtype and D must match the round's first issue");
  if (injected(ctx)) return COLI_E_INJECTED;
  cudaSetDevice(ctx->device);
  const int D = ctx->table_D;
  if (ctx->n_issued == 0) {
    int rc = ensure_slots(ctx, (size_t)COLI_MAX_ISSUES * S * D * sizeof(float));
    if (rc != COLI_OK) return rc;
    ctx->round_S = S;
    ctx->round_D = D;
    ctx->round_dtype = x_dtype;
  }
  float* slot = ctx->slots + (size_t)ctx->n_issued * S * D;
  int rc = launch_expert_group(ctx, x_rows, x_dtype, S, idx, w, n_sel, K, nullptr, slot, COLI_DTYPE_F32);
  if (rc != COLI_OK) return rc;
  ctx->compute_calls++;
  return ctx->n_issued++;
}

int coli_expert_group_take(coli_ctx* ctx, const void* resid, void* y) {
  if (!ctx) return COLI_E_INVAL;
  if (!y) return fail(ctx, COLI_E_INVAL, "take: NULL pointer");
  if (ctx->n_issued == 0) return fail(ctx, COLI_E_INVAL, "take: nothing issued");
  if (injected(ctx)) return COLI_E_INJECTED;
  cudaSetDevice(ctx->device);
  int rc = launch_take(ctx, ctx->round_S, ctx->round_D, ctx->n_issued, resid, ctx->round_dtype, y);
  if (rc != COLI_OK) return rc;
  ctx->compute_calls++;
  ctx->n_issued = 0;
  return COLI_OK;
}

}  // extern "C"
