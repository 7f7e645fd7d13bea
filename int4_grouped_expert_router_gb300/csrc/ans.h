// Compressed expert tier: the block codec (ans.cu). Declared outside the expert kernels' internal header.
#pragma once

#include <vector>

#include "coli_internal.h"

namespace coli {

constexpr uint32_t kAnsBlockBytes = 4096;  // raw bytes per independently decodable block

int ans_encode(const uint8_t* in, uint64_t n, std::vector<uint8_t>& out);  // host encoder (always succeeds)
int ans_blocks(const void* blob_host);                               // block count of an encoded stream
int launch_ans_decode(coli_ctx* ctx, const uint8_t* blob, int blocks, uint8_t* out);

// Library-owned compressed streams of a context (coli_ans_upload handles), freed with the context.
struct AnsStream {
  uint8_t* d_blob = nullptr;
  uint64_t stored = 0, raw = 0;
  int blocks = 0;
};
std::vector<AnsStream>& ans_streams(coli_ctx* ctx);
// y = resid + W x for an int4 tensor W [O x I] kept as a compressed stream (fused block decode + GEMV)
int launch_ans_gemv(coli_ctx* ctx, const AnsStream& st, const float* scales, int O, int I, int gs, const void* x,
                    int x_dtype, const void* resid, void* y);
void ans_release_all(coli_ctx* ctx);

}  // namespace coli
