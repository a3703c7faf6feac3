// Internal launch interface between the C-ABI layer (kq_api.cu) and the kernels.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include <string>

#include "kq.h"

namespace kq {

constexpr int kMaxGemvSmem = 96 * 1024;
constexpr int kSmemCap = 227 * 1024;  // opt-in shared memory per CTA on sm_103a

struct GemvPlan {
  int units = 0;        // K / 256
  int ks = 1;           // K-split across a cluster
  int chunk_units = 1;  // activation staging granularity (units)
  int grid = 0;         // CTAs
};

// Work split of the tensor-core GEMV: a function of (N, K, SM count) only.
GemvPlan plan_gemv_mma(int N, int K, int num_sms);

// Work split of the streaming (bulk-copy) GEMV; ok == false when K is too long for it.
struct TmaPlan {
  bool ok = false;
  int units = 0, tiles = 0;  // K / 256, ceil(N / 16)
  int C = 1;                 // CTAs per cluster = K-split
  int G = 0;                 // clusters
  int max_tiles = 0;         // tiles per cluster (upper bound)
};
TmaPlan plan_gemv_tma(int fmt, int N, int K, int num_sms);

// Reads and clears the device error word (bit 0: a bounded wait in a kernel gave up).
unsigned int take_device_errors(std::string* err);
size_t gemv_mma_smem(const GemvPlan& pl, int M);

// Epilogue of the streaming GEMV for the decode step's glue (fused into the GEMV's stores):
//  kind 1 (GQA expand): y as usual, and each row n of [v0, v0 + vn) is also written as bf16 to
//         out[tok][(h * group + i) * hd + d], i < group, with h = (n - v0) / hd, d = (n - v0) % hd
//         (out rows out_w wide): the attention stand-in's output feeding Wo;
//  kind 2 (SwiGLU): W's rows pair up (row i is a gate row, row N/2 + i its up row; each 16-row tile
//         takes 8 of each); out[tok][i] = bf16(silu(y_i) * y_(N/2+i)), rows N/2 wide; y is written
//         only if not null;
//  kind 3 (KV append): y as usual, and rows [v0, v0 + hd) / [v0 + hd, v0 + 2 hd) also go as bf16
//         to row row0 + tok of out / out_b (rows hd wide): the window's k and v into the cache.
struct GemvEpilogue {
  int kind = 0;
  uint16_t* out = nullptr;
  int v0 = 0, vn = 0, hd = 1, group = 1, out_w = 0;
  uint16_t* out_b = nullptr;  // kind 3: the second destination (v rows)
  int row0 = 0;               // kind 3: the first destination row (tokens go to row0 + j)
};
// Whether the streaming kernel runs this shape with this epilogue kind (kind 2 needs a plan
// without a K-split and N a multiple of 16).
bool gemv_epilogue_ok(int fmt, int N, int K, int kind, int num_sms);

// bf16 activations, tensor-core path. Returns 0 or -1 with *err set.
// overlap: launch with programmatic stream serialization (the caller guarantees the
// previous kernel in the stream does not write w). epi: null or a fused epilogue.
int launch_gemv_mma(int fmt, const void* w, const void* x, float* y, int M, int N, int K,
                    long long row_bytes, int num_sms, cudaStream_t stream, bool overlap, std::string* err,
                    const GemvEpilogue* epi = nullptr);

// Q6_K with bf16 activations, CUDA-core path (its rows are only 2-byte aligned).
int launch_gemv_q6k_bf16(const void* w, const uint16_t* x, float* y, int M, int N, int K, long long row_bytes,
                         cudaStream_t stream, bool overlap, std::string* err);

// fp32 activations, CUDA-core path.
int launch_gemv_f32(int fmt, const void* w, const float* x, float* y, int M, int N, int K,
                    long long row_bytes, cudaStream_t stream, bool overlap, std::string* err);

// Tensor-core prefill (gemm_tc.cu): Q4_K weights x bf16 activations, M > 16.
size_t gemm_tc_workspace(int M, int N, int K);
int launch_gemm_tc(const void* w, const void* x, float* y, int M, int N, int K, long long row_bytes, void* ws,
                   int num_sms, cudaStream_t stream, std::string* err);
unsigned int take_tc_errors();

// Decode step (decode.cu).
int decode_check(const kq_decode_model* m, int M, std::string* err);
size_t decode_workspace_size(const kq_decode_model* m, int M);
// The step with attention over a KV cache (decode.cu): the window's k, v are appended to
// the cache at positions L..L+M-1 of every layer.
size_t decode_attn_workspace_size(const kq_decode_model* m, int M, int L);
int decode_step_attn(const kq_decode_model* m, const kq_kv_cache* c, const uint16_t* x, float* logits, int M,
                     const uint32_t* mask, void* ws, int num_sms, cudaStream_t s, std::string* err);
// trace: null, or decode_trace_size(m, M) bytes that receive a copy of every op's output
int decode_step(const kq_decode_model* m, const uint16_t* x, float* logits, int M, void* ws, int num_sms,
                cudaStream_t s, std::string* err, void* trace = nullptr);
size_t decode_trace_size(const kq_decode_model* m, int M);

// Decode attention of a verify window over a KV cache (attention.cu).
size_t attention_workspace(int M, int L, int n_q, int n_kv, int hd);
// q rows q_stride elements apart; the output goes to o (fp32) and/or o16 (bf16), either may be null.
// early: launch the first kernel as a programmatic dependent of the previous one in the stream
// (it waits for it before its first memory access).
int launch_attention(const float* q, int q_stride, const uint16_t* k, const uint16_t* v, float* o, uint16_t* o16,
                     int M, int L, int n_q, int n_kv, int hd, const uint32_t* mask, float scale, void* ws,
                     cudaStream_t s, bool early, std::string* err);

// Shortlist output head (shortlist.cu; the small copy's build is in quantize.cu).
size_t shortlist_small_bytes(int N, int K);
size_t shortlist_bytes(int N, int K);
size_t head_argmax_workspace(int M, int N);
int launch_shortlist_build(const void* wq, void* small, float* bound, int N, int K, cudaStream_t stream,
                           std::string* err);
// The bounds and exact passes; the small-copy GEMV into the workspace's first M*N floats is
// launched before by the caller (unless all_rows).
int launch_head_select(const void* wq, const void* shortlist, bool x_bf16, const void* x, int M, int N, int K,
                       int* token, float* score, unsigned int* scored, void* ws, bool all_rows, int num_sms,
                       cudaStream_t s, std::string* err);

// GPU quantizers (fp64 arithmetic).
int launch_quantize(int fmt, const float* w, void* blocks, int N, int K, cudaStream_t stream,
                    std::string* err);

}  // namespace kq
