// Internal declarations shared by the translation units of libcoli_moe.so (not installed).
#pragma once

#include <cuda.h>  // CUtensorMap (types only; the driver entry point is fetched at run time)
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "coli_moe.h"

namespace coli {

// ---------------------------------------------------------------------------------------------
// Device-side tensor and expert descriptors
// ---------------------------------------------------------------------------------------------

// Rows per TMA box: one pipeline stage of one warp covers kBoxRows rows of its column slice.
constexpr int kBoxRows = 4;
// Words (uint32) of a row one warp owns: 32 lanes x 16 bytes.
constexpr int kSliceWords = 128;
// Chunk-group scales of one warp's slice that travel by TMA (group sizes 64..256).
constexpr int kScaleBox = 16;
// Tensor-core (prefill) weight tiles: 128 rows x 256 columns (32 words = 128 bytes of packed
// nibbles per row, staged with the 128-byte swizzle), four 64-column K tiles of the MMA.
constexpr int kTcRows = 128;
constexpr int kTcWords = 32;
// One-launch decode FFN: a work unit is kPanelCols rows of gate/up and the same columns of down.
constexpr int kPanelCols = 16;
// One-launch router scratch (router.cu): a launch counter (256 bytes), then 64-bit tagged partial
// logits of at most 15 tokens x 1024 (column part, expert) pairs.
constexpr size_t kRouterScratchBytes = 256 + (size_t)15 * 1024 * 8;

// Device status words of a context: [0] error code, [1] unused, [2..] the opt-in fused decode
// kernel's synchronisation words (grid barrier at [2], [3]; row-range counters from
// [2 + kSyncRanges]). All start at zero, and the grid barrier's count only grows.
constexpr int kSyncBase = 2;
constexpr int kSyncRanges = 64;   // offset of the range counters from kSyncBase
constexpr int kMaxRanges = 4096;  // range counters
constexpr size_t kStatusBytes = (size_t)(kSyncBase + kSyncRanges + kMaxRanges) * sizeof(int);
// The fused decode kernel covers I <= 32 * 32 * kFusedMaxSlices (column slices of a down row).
constexpr int kFusedMaxSlices = 4;

// One uploaded int4 tensor as the kernels see it. Rows are padded to a whole number of 16-byte
// chunks (32 columns each); padding nibbles hold 8, i.e. the value 0.
struct TensorDesc {
  CUtensorMap map_w;   // 2-D map over the weights as uint32 [rows x pitch/4], box [box_rows x box_w]
  CUtensorMap map_s;   // 2-D map over chunk-group scales f32 [rows x G], box [box_rows x box_s]
  CUtensorMap map_tc;  // 2-D map over the weights as uint32 [rows x pitch/4], box [kTcRows x kTcWords], 128B swizzle
  const uint8_t* w;    // rows x pitch bytes
  const float* s;      // scales: rows (gs == 0) or rows * G (gs > 0)
  uint32_t pitch;      // bytes per row, multiple of 16
  int32_t gs;          // 0 or even
  int32_t G;           // groups per row (1 when gs == 0)
  int32_t rows, cols;
  int32_t mode;        // SCALE_ROW, SCALE_CHUNK (gs % 32 == 0) or SCALE_GENERIC
  uint32_t box_rows;   // rows of a weight box (min(kBoxRows, rows))
  uint32_t box_w;      // words of a weight box row (min(kSliceWords, pitch / 4))
  uint32_t box_s;      // floats of a scale box row (0: scales are not staged by TMA)
  uint32_t pad_;
  // Panel-major view for the one-launch decode FFN (built for down tensors of the expert table,
  // NULL otherwise): column block p of kPanelCols columns is [rows x kPanelCols / 2 bytes] at
  // panel + p * rows * kPanelCols / 2; sT holds chunk-group scales transposed, [G x rows].
  const uint8_t* panel;
  const float* sT;
};

enum { SCALE_ROW = 0, SCALE_CHUNK = 1, SCALE_GENERIC = 2 };
enum { T_GATE = 0, T_UP = 1, T_DOWN = 2 };

struct ExpertDesc {
  TensorDesc t[3];
  int32_t valid;
  int32_t pad_[15];
};

// ---------------------------------------------------------------------------------------------
// Host-side context
// ---------------------------------------------------------------------------------------------

struct HostTensor {
  uint8_t* w = nullptr;
  float* s = nullptr;
  int O = 0, I = 0, gs = 0, G = 1;
  uint32_t pitch = 0;
  int table_refs = 0;
  bool live = false;
  TensorDesc desc{};  // device view, tensor maps included
  ExpertDesc* d_solo = nullptr;  // device entry {down = this tensor, valid}: the one-token dense projection
  uint8_t* panel = nullptr;      // panel-major copy (desc.panel), built when first used as a down tensor
  float* sT = nullptr;           // transposed chunk-group scales (desc.sT)
};

struct Workspace {
  char* base = nullptr;
  size_t bytes = 0;
};

}  // namespace coli

struct coli_ctx {
  int device = 0;
  cudaStream_t stream = nullptr;
  int num_sms = 0;
  std::string last_error;
  int last_code = 0;
  std::vector<coli::HostTensor> tensors;  // handle = index + 1
  // expert table
  coli::ExpertDesc* d_table = nullptr;       // COLI_MAX_EXPERTS entries
  std::vector<coli::ExpertDesc> h_table;
  std::vector<uint64_t> table_handles;       // 3 per entry
  int table_D = 0, table_I = 0, table_count = 0;
  int* d_status = nullptr;  // kStatusBytes of device status words (see kSyncBase)
  int32_t* d_solo_route = nullptr;  // device {expert 0} and, after it, {weight 1.0f}: the one-slot route
  // decode (S == 1) expert FFN as one cooperative kernel: COLI_DECODE_FUSED=1 (default 0), and how
  // this device launches it (2: cooperative + programmatic dependent launch, 1: cooperative, 0: no)
  bool decode_fused = false;
  int coop_mode = -1;  // -1: not probed yet
  // S == 1 streaming FFN (decode.cu): on unless COLI_DECODE_STREAM=0; table entries whose tensors it
  // cannot stream (group sizes that are not multiples of 32, shapes off its grid)
  bool stream_ffn = true;
  int table_nostream = 0;
  std::vector<char> table_stream;  // per entry: 1 if set and streamable, or unset
  int table_gu_maxG = 0;           // most chunk groups per gate/up row of any entry set since creation
  // test hooks read at coli_init: a shorter limit for the streaming kernel's bounded waits
  // (COLI_TEST_WAIT_NS) and, for the next N of its launches, a CTA whose producer withholds the copy
  // of its first stage so that the waits on it give up (COLI_TEST_WITHHOLD=N)
  unsigned long long wait_ns = 0;
  int test_withhold = 0;
  // the one-launch router: its scratch (kRouterScratchBytes, zeroed at creation), the rows and
  // column parts of its CTAs when set (COLI_ROUTER_ROWS, COLI_ROUTER_PARTS; 0: chosen per call),
  // and a test hook: for the next N launches its last CTA withholds token 0's partial logits, so
  // that the selection's bounded wait gives up (COLI_TEST_WITHHOLD_ROUTER=N)
  void* d_router = nullptr;
  int router_rows = 0, router_parts = 0;
  int test_withhold_router = 0;
  coli::Workspace ws;
  // resident issue/take: f32 partial sums [COLI_MAX_ISSUES][S x D] of the current round's issues
  float* slots = nullptr;
  size_t slot_bytes = 0;
  int n_issued = 0, round_S = 0, round_D = 0, round_dtype = 0;
  // COLI_FAIL_AFTER test hook
  long long fail_after = -1;
  long long compute_calls = 0;
  // per-kernel event profiling (coli_profile_enable)
  bool prof = false;
  struct ProfRec {
    int kind;
    cudaEvent_t a, b;
  };
  std::vector<ProfRec> prof_pending;
  std::vector<cudaEvent_t> prof_free;
  double prof_ms[5] = {0, 0, 0, 0, 0};
  long long prof_n[5] = {0, 0, 0, 0, 0};
};

namespace coli {

int fail(coli_ctx* ctx, int code, const std::string& msg);
int cuda_fail(coli_ctx* ctx, cudaError_t e, const char* what);
bool injected(coli_ctx* ctx);  // COLI_FAIL_AFTER: true if this compute call must fail
int ensure_workspace(coli_ctx* ctx, size_t bytes);
int ensure_slots(coli_ctx* ctx, size_t bytes);

constexpr size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Brackets one kernel launch with profiling events when profiling is on.
struct ProfScope {
  coli_ctx* ctx;
  int kind;
  cudaEvent_t a = nullptr, b = nullptr;
  ProfScope(coli_ctx* c, int k);
  ~ProfScope();
};

// Launchers (defined in router.cu / experts.cu). Arguments already validated.
// shared >= 0: every token's row gets K + 1 slots, the shared expert placed after the kept ones.
int launch_router(coli_ctx* ctx, const void* x, int x_dtype, int S, int D, const float* Wr,
                  const float* bias, int E, int K, float topp, int norm_topk, float routed_scale, int shared,
                  int32_t* idx, float* w, int32_t* n_sel);
// Tensor-core (prefill) path of coli_expert_group: bf16 activations, many routed rows per expert.
bool prefill_eligible(const coli_ctx* ctx, const void* x, int S, int K, int x_dtype);
int launch_prefill(coli_ctx* ctx, const void* x, int S, const int32_t* idx, const float* w, const int32_t* n_sel,
                   int K, const void* resid, void* y, int y_dtype);
// TMA map over a row-major bf16 matrix [rows x cols] read in 16-row x 64-column boxes with the
// 128-byte swizzle (cols a multiple of 8).
int encode_bf16_rows_map(coli_ctx* ctx, CUtensorMap* map, void* base, long long rows, int cols);

int launch_router_noalloc(coli_ctx* ctx, const void* x, int x_dtype, int S, int D, const float* Wr,
                          const float* bias, int E, int K, float topp, int norm_topk, float routed_scale, int shared,
                          int32_t* idx, float* w, int32_t* n_sel);
// y is written in y_dtype (x_dtype for coli_expert_group; f32 for an issued partial sum); resid is read in x_dtype.
int launch_expert_group(coli_ctx* ctx, const void* x, int x_dtype, int S, const int32_t* idx,
                        const float* w, const int32_t* n_sel, int K, const void* resid, void* y, int y_dtype);
// y [S x O] = resid + W x for S tokens of the uploaded tensor T [O x I] (coli_w4_linear).
// S == 1 runs the down kernel on `solo`, a one-entry table whose down tensor is T.
int launch_linear(coli_ctx* ctx, const TensorDesc& T, const ExpertDesc* solo, const void* x, int x_dtype, int S,
                  const void* resid, void* y);
// y [S x D] (dtype) = resid + the n issued partial sums [S x D] f32, added in issue order.
int launch_take(coli_ctx* ctx, int S, int D, int n, const void* resid, int dtype, void* y);
// Streaming S == 1 expert FFN (decode.cu): eligibility, launch, and the per-tensor panel view it
// streams down tensors from (built by coli_expert_table_set).
bool stream_eligible(const coli_ctx* ctx, int S);
bool stream_tensor_ok(const HostTensor& t, bool as_down);
bool stream_linear_ok(const HostTensor& t);
int launch_stream_linear(coli_ctx* ctx, const HostTensor& t, const void* x, int x_dtype, const void* resid, void* y);
int build_stream_view(coli_ctx* ctx, HostTensor& t);
int launch_stream_ffn(coli_ctx* ctx, const void* x, int x_dtype, const int32_t* idx, const float* w,
                      const int32_t* n_sel, int K, const void* resid, void* y, int y_dtype);
// Launch with programmatic stream serialisation (the kernel may start while its predecessor in
// the stream finishes; it calls griddepcontrol.wait before reading that predecessor's output) and,
// when `coop`, as a cooperative launch (every CTA resident at once, or the launch fails).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), int grid, int block, size_t smem, cudaStream_t st, bool pdl,
                            bool coop, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    na++;
  }
  if (coop) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    na++;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Which cooperative launch forms this device accepts (coli_ctx::coop_mode), found with an empty
// kernel on a private stream.
int probe_coop_mode(coli_ctx* ctx);

}  // namespace coli

// ---------------------------------------------------------------------------------------------
// Small device helpers
// ---------------------------------------------------------------------------------------------
#ifdef __CUDACC__
namespace coli {

__device__ __forceinline__ void set_error(int* err, int code) { atomicCAS(err, 0, code); }

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0;  // NaN
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// Activations may be the output of the kernel just before (programmatic dependent launch), so
// they are read through L2 (ld.global.cg), never through the non-coherent read-only path.
__device__ __forceinline__ float load_act(const void* p, int dtype, size_t i) {
  return dtype == COLI_DTYPE_F32 ? __ldcg(reinterpret_cast<const float*>(p) + i)
                                 : bf16_to_f32(__ldcg(reinterpret_cast<const unsigned short*>(p) + i));
}

// Streaming 16-byte load of packed weights: read-only, no L1 allocation, 256-byte L2 sector
// prefetch (weights are read once per call).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace coli
#endif
