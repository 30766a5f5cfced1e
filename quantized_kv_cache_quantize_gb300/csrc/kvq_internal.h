// Host-side declarations shared by the translation units of libkvq.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

// Geometry of one cache, validated once per call.
struct Geometry {
  int bh;          // batch * heads
  int d;           // head dim
  int bits;
  int group;
  int g;           // groups per token (d / group)
  int cap;         // tokens per head
  int code_bytes;  // packed bytes per token
};

// Arguments of the quantize-append kernel.
struct QuantArgs {
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint8_t* k_codes;
  uint8_t* v_codes;
  uint32_t* k_sz;  // one 32-bit word (bf16 step | bf16 zero << 16) per group
  uint32_t* v_sz;
  int bh;
  int n_new;
  int cap;
  int first;       // first token written in every head
  uint32_t sign_bits[4];
  float inv_sqrt_d;
};

// Arguments of the rotation kernel: up to three row segments in one launch.
struct RotateArgs {
  const uint16_t* src[3];
  void* dst[3];
  long long rows[3];
  uint32_t sign_bits[4];
  float inv_sqrt_d;
  int out_f32;  // 1: fp32 output, 0: fp16 (the attention kernel's operand format)
};

cudaError_t launch_quantize_append(const QuantArgs& a, int d, int bits, int group,
                                   cudaStream_t stream, bool* supported);
cudaError_t launch_rotate(const RotateArgs& a, int d, cudaStream_t stream);

// Attention ---------------------------------------------------------------

struct AttnLaunch {
  // cache
  const uint8_t* k_codes;
  const uint8_t* v_codes;
  const uint32_t* k_sz;
  const uint32_t* v_sz;
  int n_s;   // valid cached tokens per head
  int cap;
  // rotated current-chunk tensors (workspace)
  const uint16_t* q_rot;
  const uint16_t* k_rot;
  const uint16_t* v_rot;
  int n_q, n_r, bh;
  float scale;
  int corr;
  int mass_only;
  uint16_t* out;
  float* p_s;
  float* p_r;
  uint32_t sign_bits[4];
  unsigned long long wait_limit_ns;
};

kvq_status launch_attention(const AttnLaunch& a, int d, int bits, int group,
                            cudaStream_t stream);
kvq_status read_and_clear_attention_status(int* status);
cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t stream);

}  // namespace kvq
