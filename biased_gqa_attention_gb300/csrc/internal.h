// internal.h -- launchers shared between the extkv translation units (host side).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "extkv.h"

namespace extkv {

struct BiasSpec;  // common.cuh

struct AttnArgs {
  void* y;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const void* bias;       // materialised bias or nullptr
  const void* extra;      // fused spec's extra term or nullptr
  const int64_t* span_offsets;
  const int64_t* spans;
  const int64_t* q_start;
  int32_t causal, window;
  int fused;              // evaluate the spec in registers
  const int64_t* nonpad;
  float scale;
  float softcap;  // > 0: scores capped to softcap * tanh(score / softcap) before the bias
  int64_t B, Hq, Hkv, S_q, max_seq, D;  // D: head size of q and k
  int64_t Dv;                            // head size of v and y (== D unless asymmetric)
  int dtype;
  int32_t* status;
  void* workspace;
  size_t ws_bytes;
  cudaStream_t stream;
  // fused scatter, taken by the decode kernel (k_new == nullptr: none)
  void* kc_w;
  void* vc_w;
  const void* k_new;
  const void* v_new;
  const int64_t* write_idx;
  int64_t S_new;
  // limit of the pipeline's barrier waits: 0, the kernels' own limit; n + 1,
  // n polls (a test sets a tiny one to make the waits run out)
  uint32_t wait_limit_plus1;
  // 1: the prefill at head size 256 may run on CTA pairs (2-SM MMAs); 0: one
  // CTA per query tile only
  int prefill_pairs;
  // which decode kernel takes a decode call: kDecodeAuto (by shape),
  // kDecodeStreamK (plan, stream-K decode, merge) or kDecodeCluster (one
  // cluster per KV head, one kernel)
  int decode_variant;
};

constexpr int kDecodeAuto = 0, kDecodeStreamK = 1, kDecodeCluster = 2;

// Each launcher returns cudaSuccess or the launch error; `name` receives the
// kernel's name for extkv_last_kernel().
cudaError_t launch_scatter(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                           const int64_t* write_idx, int64_t B, int64_t Hkv, int64_t S_new,
                           int64_t max_seq, int64_t D, int dtype, int32_t* status,
                           cudaStream_t stream);
cudaError_t launch_bias(void* bias, const extkv_bias_spec& spec, const int64_t* nonpad, int64_t B,
                        int64_t S_q, int64_t max_seq, int dtype, int32_t* status,
                        cudaStream_t stream);
cudaError_t launch_mask_bias(void* bias, const uint8_t* mask, int64_t n, int dtype, cudaStream_t stream);
cudaError_t launch_attn_generic(const AttnArgs& a, const char** name);

// Fast paths: `supported` says whether the shape can run; launch returns the error.
bool decode_supported(const AttnArgs& a);
size_t decode_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t S_q, int64_t max_seq, int64_t Dk,
                              int64_t Dv);
cudaError_t launch_attn_decode(const AttnArgs& a, const char** name);
// The cluster decode kernel: CTAs per cluster it would use for this call (0:
// it cannot take the call), clusters per unit (M > 1: each cluster leaves a
// partial for the stream-K merge kernel), and its launch.
int decode_cluster_size(const AttnArgs& a);
int decode_cluster_split(const AttnArgs& a, int C);
cudaError_t launch_attn_decode_cluster(const AttnArgs& a, int C, int M, const char** name);
bool prefill_supported(const AttnArgs& a);
// Dk, Dv: the key and value head sizes (the partial rows of key splits hold Dv columns)
size_t prefill_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t S_q, int64_t max_seq, int64_t Dk,
                               int64_t Dv, bool term);
cudaError_t launch_attn_prefill(const AttnArgs& a, const char** name);

int num_sms();

// Sets the calling thread's extkv_last_error() message.
void set_error(const char* msg);

// Records how many kernels the attention launcher just launched (read back
// through extkv_last_launches()).
void note_launches(int n);

// The calling thread's extkv_set_wait_polls() setting, as AttnArgs::wait_limit_plus1.
uint32_t wait_limit_setting();

// The poll limit of a pipeline wait for a call's wait_limit_plus1.
inline uint32_t wait_limit(uint32_t plus1, uint32_t own) { return plus1 ? plus1 - 1 : own; }

// Records a successful attention call made outside attention_ext_kv's own
// dispatch: extkv_last_kernel() then names `name`, and extkv_last_launches()
// the count the launcher noted.
void note_last_call(const char* name);

}  // namespace extkv
