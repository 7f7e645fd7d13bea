// Expert parallelism across GPUs, the device half (see ep.h).
//
// Experts are owned by rank e mod world. Every rank runs the same router, keeps the routes of its own
// experts (routes_shard_kernel), computes their weighted slot-order sum without the residual, and the
// ranks' partial rows are then gathered and added in rank order with the residual last
// (partials_reduce_kernel): a deterministic fixed-order reduce with no atomics, as PR #434
// "COLI_CUDA_RESID=1", section "What", reduces the per-device partial sums of the expert groups that the
// "GPU resident pipeline" commit of the c/backend_cuda.cu history spreads over the cards. Against one GPU
// the result differs only in how the slots' terms are grouped before rounding.
#include "ep.h"

namespace coli {

// One warp per token: a ballot of the lanes whose kept slot belongs to this rank, and each such lane
// writes its route to the position given by the count of owned slots before it.
__global__ void routes_shard_kernel(const int32_t* __restrict__ idx, const float* __restrict__ w,
                                    const int32_t* __restrict__ n_sel, int S, int K, int rank, int world,
                                    int32_t* __restrict__ idx_out, float* __restrict__ w_out,
                                    int32_t* __restrict__ n_out, int* err) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= S) return;  // uniform per warp
  int n = n_sel ? n_sel[t] : K;
  n = n < 0 ? 0 : (n > K ? K : n);
  const bool kept = lane < n;
  const int e = kept ? idx[(size_t)t * K + lane] : -1;
  const float wv = kept ? w[(size_t)t * K + lane] : 0.f;
  if (kept && (e < 0 || e >= COLI_MAX_EXPERTS)) set_error(err, COLI_E_ROUTE);
  const bool mine = kept && e >= 0 && e < COLI_MAX_EXPERTS && e % world == rank;
  const unsigned own = __ballot_sync(0xffffffffu, mine);
  const int cnt = __popc(own);
  if (mine) {
    const int pos = __popc(own & ((1u << lane) - 1u));
    idx_out[(size_t)t * K + pos] = e;
    w_out[(size_t)t * K + pos] = wv;
  }
  if (lane < K && lane >= cnt) {
    idx_out[(size_t)t * K + lane] = -1;
    w_out[(size_t)t * K + lane] = 0.f;
  }
  if (lane == 0) n_out[t] = cnt;
}

__global__ void partials_reduce_kernel(const float* __restrict__ parts, int n, long long cells, const void* resid,
                                       int dtype, void* y) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < cells; i += (long long)gridDim.x * blockDim.x) {
    float acc = parts[i];
    for (int r = 1; r < n; r++) acc = acc + parts[(size_t)r * cells + i];
    if (resid) acc = load_act(resid, dtype, (size_t)i) + acc;
    if (dtype == COLI_DTYPE_F32)
      static_cast<float*>(y)[i] = acc;
    else
      static_cast<uint16_t*>(y)[i] = f32_to_bf16_rn(acc);
  }
}

int launch_routes_shard(coli_ctx* ctx, const int32_t* idx, const float* w, const int32_t* n_sel, int S, int K,
                        int rank, int world, int32_t* idx_out, float* w_out, int32_t* n_out) {
  const int warps = 8;
  routes_shard_kernel<<<(S + warps - 1) / warps, warps * 32, 0, ctx->stream>>>(idx, w, n_sel, S, K, rank, world, idx_out,
                                                                              w_out, n_out, ctx->d_status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(ctx, e, "routes_shard launch");
  return COLI_OK;
}

int launch_partials_reduce(coli_ctx* ctx, const float* parts, int n, int S, int D, const void* resid, int dtype,
                           void* y) {
  const long long cells = (long long)S * D;
  long long grid = (cells + 255) / 256;
  if (grid > 4LL * ctx->num_sms) grid = 4LL * ctx->num_sms;
  ProfScope prof(ctx, COLI_KERNEL_COMBINE);
  partials_reduce_kernel<<<(int)grid, 256, 0, ctx->stream>>>(parts, n, cells, resid, dtype, y);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(ctx, e, "partials_reduce launch");
  return COLI_OK;
}

}  // namespace coli
