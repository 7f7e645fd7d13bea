// The int4 x activation dot product shared by the expert kernels.
//
// A thread owns a block of N consecutive columns of a weight row (N = 32: one 16-byte chunk; N = 16:
// 8 bytes) and keeps the matching N activations in registers in block-fixed-point form: the block
// is scaled by a power of two 2^q so that its largest magnitude lies in [2^21, 2^22), rounded to
// integers and split into three balanced signed bytes (x = l2 2^16 + l1 2^8 + l0). The
// nibble-by-limb products are then summed exactly in 32-bit integers with dp4a (four products per
// instruction), the offset 8 is removed through a precomputed -8 * sum(l), and the exact limb sums
// are combined in binary32 and scaled back by 2^-q. The block result therefore differs from the
// exact dot product of the given activations by two roundings of binary32 plus the activation
// quantisation: at most 2^-22 of the block's largest activation, per column.
//
// Stored format (c/backend_cuda.cu commit history, commit "grouped MoE kernels were per-row-only"):
// offset-8 nibbles, column 2m in the low nibble of byte m and column 2m + 1 in its high nibble.
#pragma once

#include "coli_internal.h"
#include "pipe.h"

namespace coli {

// Limbs of a block of 8 NWD columns: NWD 32-bit words of packed nibbles per block row.
template <int NWD>
struct LimbsN {
  uint32_t r[NWD][2][3];  // [32-bit word of the block][even/odd columns][limb]: 4 bytes each
  int32_t a0[3];          // even-column accumulator start: -8 * sum over the even columns of limb l
  int32_t b0[3];          // odd-column accumulator start: -128 * sum over the odd columns of limb l
  float k01, k2;          // 2^(-q-4) and 2^(16-q-4)
};
using Limbs = LimbsN<4>;    // 32 columns, one 16-byte chunk
using Limbs16 = LimbsN<2>;  // 16 columns, 8 bytes

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// v[j] = activation of column j of the block (0 beyond the matrix). Returns false if any is not
// finite. Balanced base-256 digits: for |X| < 2^23 - 2^15 the bytes of Y = X + 0x808080 are the
// digits l_k + 128 (each in [0, 255], so no carries), hence the bytes of Y ^ 0x808080 are the signed
// digits l_0, l_1, l_2 with X = l_2 2^16 + l_1 2^8 + l_0.
template <int N>
__device__ __forceinline__ bool make_limbs(const float (&v)[N], LimbsN<N / 8>& L) {
  static_assert(N % 8 == 0, "blocks of whole 32-bit words");
  float M = 0.f, nan_probe = 0.f;
#pragma unroll
  for (int j = 0; j < N; j++) {
    M = fmaxf(M, fabsf(v[j]));
    nan_probe = fmaf(v[j], 0.f, nan_probe);  // NaN once any v is NaN or infinite
  }
  const bool finite = nan_probe == 0.f;
  int e = 0;
  if (finite && M > 0.f) frexpf(M, &e);  // M < 2^e
  int q = 22 - e;                         // M 2^q in [2^21, 2^22)
  q = q > 122 ? 122 : q;                  // 2^(-q-4) stays a normal float (|x| < 2^-100 only)
  const float scale = (finite && M > 0.f) ? __int_as_float((127 + q) << 23) : 0.f;  // 2^q, q in [-107, 122]
  uint32_t z[N];
#pragma unroll
  for (int j = 0; j < N; j++) {
    const int xi = __float2int_rn(v[j] * scale);  // exact scaling by a power of two; |xi| <= 2^22
    z[j] = ((uint32_t)xi + 0x808080u) ^ 0x808080u;
  }
  // word w, parity p, limb l: byte b is limb l of column 8 w + 2 b + p
#pragma unroll
  for (int w = 0; w < N / 8; w++)
#pragma unroll
    for (int p = 0; p < 2; p++) {
      const uint32_t z0 = z[8 * w + p], z1 = z[8 * w + 2 + p], z2 = z[8 * w + 4 + p], z3 = z[8 * w + 6 + p];
      const uint32_t a01 = prmt(z0, z1, 0x5140u);  // z0.b0 z1.b0 z0.b1 z1.b1
      const uint32_t a23 = prmt(z2, z3, 0x5140u);
      const uint32_t c01 = prmt(z0, z1, 0x6262u);  // z0.b2 z1.b2 (twice)
      const uint32_t c23 = prmt(z2, z3, 0x6262u);
      L.r[w][p][0] = prmt(a01, a23, 0x5410u);
      L.r[w][p][1] = prmt(a01, a23, 0x7632u);
      L.r[w][p][2] = prmt(c01, c23, 0x5410u);
    }
#pragma unroll
  for (int l = 0; l < 3; l++) {
    int se = 0, so = 0;
#pragma unroll
    for (int w = 0; w < N / 8; w++) {
      se = dp4a_ss(L.r[w][0][l], 0x01010101u, se);
      so = dp4a_ss(L.r[w][1][l], 0x01010101u, so);
    }
    L.a0[l] = -8 * se;
    L.b0[l] = -128 * so;
  }
  L.k01 = (finite && M > 0.f) ? __int_as_float((127 - q - 4) << 23) : 0.f;
  L.k2 = (finite && M > 0.f) ? __int_as_float((127 + 12 - q) << 23) : 0.f;
  return finite;
}

// sum_j (n_j - 8) x_j over the 8 NWD columns of one block, n_j the stored nibbles in wv.
// Even columns (low nibbles, w & 0x0f0f0f0f) and odd columns (high nibbles kept in place,
// w & 0xf0f0f0f0 = 16 n) accumulate in separate dp4a chains; t_l = 16 a_l + b_l is then 16 times
// the exact limb sum sum_j (n_j - 8) l_j (|t_l| < 2^19). Limbs 0 and 1 are joined exactly in
// 32-bit integers, t_0 + 256 t_1 (below 2^28); that and t_2 are converted once each and scaled by
// powers of two: the result is the dot product with the quantised activations, rounded twice.
template <int NWD>
__device__ __forceinline__ float block_dot(const uint32_t (&words)[NWD], const LimbsN<NWD>& L) {
  int a0 = L.a0[0], a1 = L.a0[1], a2 = L.a0[2];
  int b0 = L.b0[0], b1 = L.b0[1], b2 = L.b0[2];
#pragma unroll
  for (int w = 0; w < NWD; w++) {
    const uint32_t lo = words[w] & 0x0f0f0f0fu;  // even columns: n
    const uint32_t hi = words[w] & 0xf0f0f0f0u;  // odd columns: 16 n
    a0 = dp4a_us(lo, L.r[w][0][0], a0);
    a1 = dp4a_us(lo, L.r[w][0][1], a1);
    a2 = dp4a_us(lo, L.r[w][0][2], a2);
    b0 = dp4a_us(hi, L.r[w][1][0], b0);
    b1 = dp4a_us(hi, L.r[w][1][1], b1);
    b2 = dp4a_us(hi, L.r[w][1][2], b2);
  }
  const int t0 = 16 * a0 + b0, t1 = 16 * a1 + b1, t2 = 16 * a2 + b2;
  const int p01 = t0 + 256 * t1;
  return fmaf(__int2float_rn(t2), L.k2, __int2float_rn(p01) * L.k01);
}

__device__ __forceinline__ float chunk_dot(const uint4 wv, const Limbs& L) {
  const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
  return block_dot<4>(words, L);
}

__device__ __forceinline__ float chunk_dot16(const uint2 wv, const Limbs16& L) {
  const uint32_t words[2] = {wv.x, wv.y};
  return block_dot<2>(words, L);
}

// Any even gs that is not a multiple of 32: a chunk may cross group boundaries, so each column
// takes its own group's scale (binary32 products and sums, columns in order). The activations are
// re-read from memory (act[base + col]). Returns the scaled partial sum.
static __device__ __noinline__ float chunk_dot_generic(const uint4 wv, const void* act, int dtype, size_t base,
                                                const TensorDesc* T, int row, int c) {
  const int gs = T->gs, G = T->G, cols = T->cols;
  const float* srow = T->s + (size_t)row * G;
  const int col0 = 32 * c;
  int g = col0 / gs;
  int next = (g + 1) * gs;
  float acc = 0.f;
  for (int j = 0; j < 32; j++) {
    const int col = col0 + j;
    if (col >= cols) break;
    if (col >= next) {
      g++;
      next += gs;
    }
    const uint32_t word = j < 8 ? wv.x : (j < 16 ? wv.y : (j < 24 ? wv.z : wv.w));
    const int n = (int)((word >> (4 * (j & 7))) & 0xfu) - 8;
    acc = fmaf(__ldg(srow + g) * (float)n, load_act(act, dtype, base + col), acc);
  }
  return acc;
}

// Butterfly reduction of N values per lane across the warp: afterwards lane l holds, in v[0],
// the warp total of value l / (32 / N). N - 1 + log2(32 / N) shuffles.
template <int N>
__device__ __forceinline__ void warp_transpose_reduce(float (&v)[N], int lane) {
#pragma unroll
  for (int cnt = N, off = 16; cnt > 1; cnt >>= 1, off >>= 1) {
    const bool upper = lane & off;
    const int half = cnt >> 1;
#pragma unroll
    for (int i = 0; i < half; i++) {
      float send = upper ? v[i] : v[i + half];
      float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
#pragma unroll
  for (int off = 16 / N; off > 0; off >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// v[j] = activation (f32 or bf16, widened exactly) of column col0 + j, 0 at and beyond `cols`.
// Whole chunks of aligned rows use 16-byte loads through L2.
__device__ __forceinline__ void load_chunk_f32(const void* p, int dtype, size_t base, int col0, int cols,
                                               float (&v)[32]) {
  const bool full = col0 + 32 <= cols;
  if (dtype == COLI_DTYPE_F32) {
    const float* q = static_cast<const float*>(p) + base + col0;
    if (full && (reinterpret_cast<uintptr_t>(q) & 15) == 0) {
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const float4 f = __ldcg(reinterpret_cast<const float4*>(q) + i);
        v[4 * i] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
      }
      return;
    }
  } else {
    const uint16_t* q = static_cast<const uint16_t*>(p) + base + col0;
    if (full && (reinterpret_cast<uintptr_t>(q) & 15) == 0) {
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const uint4 u = __ldcg(reinterpret_cast<const uint4*>(q) + i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int h = 0; h < 4; h++) {
          v[8 * i + 2 * h] = __uint_as_float(w[h] << 16);
          v[8 * i + 2 * h + 1] = __uint_as_float(w[h] & 0xffff0000u);
        }
      }
      return;
    }
  }
#pragma unroll
  for (int j = 0; j < 32; j++) v[j] = (col0 + j < cols) ? load_act(p, dtype, base + col0 + j) : 0.f;
}

}  // namespace coli
