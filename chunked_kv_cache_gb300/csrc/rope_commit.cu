// rope_commit.cu -- 3D (t, h, w) rotary positions on chunk tokens, fused with
// the in-place ring-buffer write of the committed keys and values.
//
// H3 project page ("Interactive Coding Worlds with Real-time Streaming
// Diffusion Render"), section 3.2 Iteration 3 item 2: a latent frame gets its
// rotary position a single time, when it is stored into a fixed slot of a ring
// allocated up front; Iteration 4: the time coordinate is the frame's absolute
// index in the stream; section 3.3 "Persistent KV layout": the cache is
// modified where it lives, never rebuilt.
//
// Work split: every thread moves 16-byte vectors (8 bf16 = 4 rotary pairs) of
// token-major [L][H][d] rows, so loads and stores are fully coalesced. The
// cos/sin of a token's d/2 pairs do not depend on the head: a CTA first fills a
// small shared-memory table for the tokens it covers, then every head reuses it.
// HBM bound: the kernel reads 2 and writes 2 tensors of L*H*d bf16 once.
#include <cuda_bf16.h>

#include "sr_kernels.h"

namespace sr {

namespace {

constexpr int kRopeThreads = 256;
constexpr int kRopeVecPerThread = 4;
constexpr int kRopeVecPerCta = kRopeThreads * kRopeVecPerThread;

__device__ __forceinline__ uint32_t rotate_pair(uint32_t packed, float c, float s) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&packed);
  const float x0 = __low2float(v);
  const float x1 = __high2float(v);
  const float y0 = fmaf(x0, c, -x1 * s);
  const float y1 = fmaf(x0, s, x1 * c);
  __nv_bfloat162 out = __floats2bfloat162_rn(y0, y1);
  return *reinterpret_cast<uint32_t*>(&out);
}

template <int D>
__global__ void __launch_bounds__(kRopeThreads) rope_kernel(const RopeParams p) {
  extern __shared__ float2 cs_table[];  // [tokens of this CTA][D/2] (cos, sin)
  constexpr int kPairs = D / 2;
  constexpr int kVecPerHead = D / 8;
  const int vec_per_tok = p.n_heads * kVecPerHead;
  const int64_t total = static_cast<int64_t>(p.n_tok) * vec_per_tok;
  const int64_t v0 = static_cast<int64_t>(blockIdx.x) * kRopeVecPerCta;
  if (v0 >= total) return;
  const int64_t v1 = min(v0 + kRopeVecPerCta, total);
  const int tok_lo = static_cast<int>(v0 / vec_per_tok);
  const int tok_hi = static_cast<int>((v1 - 1) / vec_per_tok);
  const int ntok = tok_hi - tok_lo + 1;

  // Slot table: frame g = n + f now lives in slot g mod W.
  if (p.mode == 1 && blockIdx.x == 0 && threadIdx.x < p.chunk_frames) {
    const int64_t g = p.n_committed + threadIdx.x;
    p.slot_frame[g % p.window_frames] = static_cast<int32_t>(g);
  }

  // Loads first: they are in flight while the sin/cos table is built.
  uint4 a[kRopeVecPerThread], b[kRopeVecPerThread];
  const uint4* s0 = reinterpret_cast<const uint4*>(p.src0);
  const uint4* s1 = reinterpret_cast<const uint4*>(p.src1);
#pragma unroll
  for (int k = 0; k < kRopeVecPerThread; ++k) {
    const int64_t v = v0 + threadIdx.x + k * kRopeThreads;
    if (v < v1) {
      a[k] = s0[v];
      b[k] = s1[v];
    }
  }

  // Angle = pos * inv_freq, carried as an unevaluated sum of two floats (the
  // rounded product, its exact FMA error, and pos times the low half of
  // inv_freq), then reduced by 2*pi written as two floats (Cody-Waite) before
  // the fp32 sincos. A plain fp32 product would carry an absolute error
  // proportional to the angle (1e-4 rad at t ~ 1000); this keeps it ~1e-7.
  for (int i = threadIdx.x; i < ntok * kPairs; i += kRopeThreads) {
    const int tok = tok_lo + i / kPairs;
    const int pr = i % kPairs;
    const int ax = p.axis[pr];
    const int in_frame = tok % p.tokens_per_frame;
    int64_t pos;
    if (ax == 0)
      pos = p.t_clock0 + p.n_committed + tok / p.tokens_per_frame;
    else if (ax == 1)
      pos = in_frame / p.grid_w;
    else
      pos = in_frame % p.grid_w;
    const float fp = static_cast<float>(pos);            // exact below 2^24
    const float hi = p.inv_freq_hi[pr];
    const float prod = fp * hi;
    const float err = fmaf(fp, p.inv_freq_lo[pr], fmaf(fp, hi, -prod));
    const float k = rintf(prod * 0.159154943091895336f);
    float r = fmaf(-k, 6.28318548202514648f, prod);       // 2*pi rounded to float
    r = fmaf(-k, -1.74845553146951906e-7f, r);            // 2*pi minus that float
    r += err;
    float sn, cs;
    sincosf(r, &sn, &cs);
    cs_table[i] = make_float2(cs, sn);
  }
  __syncthreads();

  uint4* d0 = reinterpret_cast<uint4*>(p.dst0);
  uint4* d1 = reinterpret_cast<uint4*>(p.dst1);
#pragma unroll
  for (int k = 0; k < kRopeVecPerThread; ++k) {
    const int64_t v = v0 + threadIdx.x + k * kRopeThreads;
    if (v >= v1) continue;
    const int tok = static_cast<int>(v / vec_per_tok);
    const int c8 = static_cast<int>(v % kVecPerHead);          // which 8-element group of the head
    const float2* cs = cs_table + (tok - tok_lo) * kPairs + c8 * 4;
    uint32_t* wa = reinterpret_cast<uint32_t*>(&a[k]);
#pragma unroll
    for (int j = 0; j < 4; ++j) wa[j] = rotate_pair(wa[j], cs[j].x, cs[j].y);
    int64_t dst = v;
    if (p.mode == 0) {
      uint32_t* wb = reinterpret_cast<uint32_t*>(&b[k]);
#pragma unroll
      for (int j = 0; j < 4; ++j) wb[j] = rotate_pair(wb[j], cs[j].x, cs[j].y);
    } else {
      // token -> ring row: frame f of the chunk goes to slot (n + f) mod W
      const int f = tok / p.tokens_per_frame;
      const int r = tok % p.tokens_per_frame;
      const int slot = static_cast<int>((p.n_committed + f) % p.window_frames);
      const int64_t row = static_cast<int64_t>(slot) * p.tokens_per_frame + r;
      dst = row * vec_per_tok + (v % vec_per_tok);
    }
    d0[dst] = a[k];
    d1[dst] = b[k];
  }
}

}  // namespace

cudaError_t launch_rope(const RopeParams& p, int head_dim, cudaStream_t st) {
  const int vec_per_tok = p.n_heads * head_dim / 8;
  const int64_t total = static_cast<int64_t>(p.n_tok) * vec_per_tok;
  if (total == 0) return cudaSuccess;
  const int64_t grid = (total + kRopeVecPerCta - 1) / kRopeVecPerCta;
  const int max_tok = kRopeVecPerCta / vec_per_tok + 2;
  const size_t smem = static_cast<size_t>(max_tok) * (head_dim / 2) * sizeof(float2);
  if (head_dim == 128) {
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(rope_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    rope_kernel<128><<<static_cast<unsigned>(grid), kRopeThreads, smem, st>>>(p);
  } else {
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(rope_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    rope_kernel<64><<<static_cast<unsigned>(grid), kRopeThreads, smem, st>>>(p);
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------ small helpers

namespace {
__global__ void copy16_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    dst[i] = src[i];
}
__global__ void init_ring_state_kernel(int32_t* slot_frame, int W, int32_t* err_word, int32_t* ws_ctr, int n_ctr) {
  for (int i = threadIdx.x; i < W; i += blockDim.x) slot_frame[i] = -1;
  if (ws_ctr)
    for (int i = threadIdx.x; i < n_ctr; i += blockDim.x) ws_ctr[i] = 0;
  if (threadIdx.x == 0) *err_word = SR_DEVERR_NONE;
}
}  // namespace

cudaError_t launch_copy16(void* dst, const void* src, size_t bytes, cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(bytes / 16);
  if (n == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 152 * 16);
  copy16_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(static_cast<uint4*>(dst),
                                                                static_cast<const uint4*>(src), n);
  return cudaGetLastError();
}

cudaError_t launch_init_ring_state(int32_t* slot_frame, int W, int32_t* err_word, int32_t* ws_ctr, int n_ctr,
                                   cudaStream_t st) {
  init_ring_state_kernel<<<1, 256, 0, st>>>(slot_frame, W, err_word, ws_ctr, n_ctr);
  return cudaGetLastError();
}

}  // namespace sr
