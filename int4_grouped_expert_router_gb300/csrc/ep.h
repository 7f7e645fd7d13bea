// Expert-parallel pieces (ep.cu): a rank's share of each token's routes, and the fixed-order sum of the
// ranks' partial rows. Declared here, outside the expert kernels' internal header, so that adding them
// leaves those kernels' sources untouched.
#pragma once

#include "coli_internal.h"

namespace coli {

// idx_out/w_out [S x K], n_out [S]: token t's kept slots (k < n_sel[t], all K if n_sel is NULL) whose
// expert e has e mod world == rank, moved to the front in slot order; the other slots -1 / 0.
int launch_routes_shard(coli_ctx* ctx, const int32_t* idx, const float* w, const int32_t* n_sel, int S, int K,
                        int rank, int world, int32_t* idx_out, float* w_out, int32_t* n_out);

// y [S x D] (dtype) = resid + (((p_0 + p_1) + p_2) + ...), the n partial rows [n x S x D] f32 in order.
int launch_partials_reduce(coli_ctx* ctx, const float* parts, int n, int S, int D, const void* resid, int dtype,
                           void* y);

}  // namespace coli
