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
// Work split: a CTA takes whole tokens (tokens_per_cta of them, up to 1024
// 16-byte vectors of each tensor), and every thread moves 16-byte vectors (8
// bf16 = 4 rotary pairs) of the token-major [L][H][d] rows, so loads and
// stores are fully coalesced. The cos/sin of a token's d/2 pairs do not depend
// on the head: the CTA fills a small shared-memory table for its tokens while
// its loads are in flight, and every head reuses it. Threads walk their
// vectors with running (token, vector) counters, so no vector pays an integer
// division. HBM bound: the kernel reads 2 and writes 2 tensors of L*H*d bf16
// once.
#include <cuda_bf16.h>

#include "sr_device.cuh"
#include "sr_kernels.h"

namespace sr {

namespace {

constexpr int kRopeThreads = 256;
constexpr int kRopeVecPerThread = 4;     // per tensor and pass
constexpr int kRopeVecTarget = kRopeThreads * kRopeVecPerThread;

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
__global__ void __launch_bounds__(kRopeThreads) rope_kernel(const RopeParams p, int tokens_per_cta) {
  constexpr int kPairs = D / 2;
  constexpr int kVecPerHead = D / 8;
  grid_dep_wait();   // the previous kernel of the stream may still be draining
  grid_dep_launch_dependents();
  extern __shared__ float2 smem_rope[];
  float2* cs_table = smem_rope;                                               // [tokens_per_cta][D/2]
  int32_t* dst_row = reinterpret_cast<int32_t*>(smem_rope + tokens_per_cta * kPairs);   // [tokens_per_cta]
  const int vpt = p.n_heads * kVecPerHead;   // vectors per token
  const int tok_lo = blockIdx.x * tokens_per_cta;
  if (tok_lo >= p.n_tok) return;
  const int ntok = min(tokens_per_cta, p.n_tok - tok_lo);
  const int nvec = ntok * vpt;
  // frames committed before this chunk: from the device counter when one is given
  const int64_t n0 = (p.dev_n != nullptr ? *p.dev_n : 0) + p.n_committed;

  // Slot table: frame g = n + f now lives in slot g mod W.
  if (p.mode == 1 && blockIdx.x == 0) {
    for (int f = threadIdx.x; f < p.chunk_frames; f += kRopeThreads) {
      const int64_t g = n0 + f;
      p.slot_frame[g % p.window_frames] = static_cast<int32_t>(g);
    }
  }

  const uint4* s0 = reinterpret_cast<const uint4*>(p.src0) + static_cast<int64_t>(tok_lo) * vpt;
  const uint4* s1 = reinterpret_cast<const uint4*>(p.src1) + static_cast<int64_t>(tok_lo) * vpt;
  uint4* d0 = reinterpret_cast<uint4*>(p.dst0);
  uint4* d1 = reinterpret_cast<uint4*>(p.dst1);

  for (int base = 0; base < nvec; base += kRopeVecTarget) {
    // Loads first: they are in flight while the sin/cos table is built.
    uint4 a[kRopeVecPerThread], b[kRopeVecPerThread];
#pragma unroll
    for (int k = 0; k < kRopeVecPerThread; ++k) {
      const int j = base + threadIdx.x + k * kRopeThreads;
      if (j < nvec) {
        a[k] = s0[j];
        b[k] = s1[j];
      }
    }

    if (base == 0) {
      // The angle of each (token, pair): the pair's fixed-point turn constant
      // times the integer position, reduced to one turn with integer
      // arithmetic (rope_angle), then the fp32 sincos of that angle in [-pi, pi).
      for (int i = threadIdx.x; i < ntok * kPairs; i += kRopeThreads) {
        const int tok = tok_lo + i / kPairs;
        const int pr = i % kPairs;
        const int ax = p.phase.axis[pr];
        const int in_frame = tok % p.tokens_per_frame;
        int64_t pos;
        if (ax == 0)
          pos = p.t_clock0 + n0 + tok / p.tokens_per_frame;
        else if (ax == 1)
          pos = in_frame / p.grid_w;
        else
          pos = in_frame % p.grid_w;
        const float r = rope_angle(p.phase.turn_hi[pr], p.phase.turn_lo[pr], pos, p.phase.rad_hi, p.phase.rad_lo);
        float sn, cs;
        sincosf(r, &sn, &cs);
        cs_table[i] = make_float2(cs, sn);
      }
      // destination row of each token: itself (mode 0) or its ring row (mode 1),
      // where frame f of the chunk goes to slot (n + f) mod W
      for (int t = threadIdx.x; t < ntok; t += kRopeThreads) {
        const int tok = tok_lo + t;
        if (p.mode == 0) {
          dst_row[t] = tok;
        } else {
          const int f = tok / p.tokens_per_frame;
          const int r = tok - f * p.tokens_per_frame;
          const int slot = static_cast<int>((n0 + f) % p.window_frames);
          dst_row[t] = slot * p.tokens_per_frame + r;
        }
      }
      __syncthreads();
    }

    // this thread's first vector: token t, vector r within the token
    int j = base + threadIdx.x;
    int t = j / vpt;
    int r = j - t * vpt;
#pragma unroll
    for (int k = 0; k < kRopeVecPerThread; ++k) {
      if (j < nvec) {
        const float2* cs = cs_table + t * kPairs + (r & (kVecPerHead - 1)) * 4;
        uint32_t* wa = reinterpret_cast<uint32_t*>(&a[k]);
#pragma unroll
        for (int q = 0; q < 4; ++q) wa[q] = rotate_pair(wa[q], cs[q].x, cs[q].y);
        if (p.mode == 0) {
          uint32_t* wb = reinterpret_cast<uint32_t*>(&b[k]);
#pragma unroll
          for (int q = 0; q < 4; ++q) wb[q] = rotate_pair(wb[q], cs[q].x, cs[q].y);
        }
        const int64_t dst = static_cast<int64_t>(dst_row[t]) * vpt + r;
        d0[dst] = a[k];
        d1[dst] = b[k];
      }
      j += kRopeThreads;
      r += kRopeThreads;
      while (r >= vpt) {
        r -= vpt;
        ++t;
      }
    }
  }
}

}  // namespace

cudaError_t launch_rope(const RopeParams& p, int head_dim, cudaStream_t st) {
  if (p.n_tok <= 0) return cudaSuccess;
  const int vpt = p.n_heads * head_dim / 8;
  const int tokens_per_cta = std::max(1, kRopeVecTarget / vpt);
  const int grid = (p.n_tok + tokens_per_cta - 1) / tokens_per_cta;
  const size_t smem = static_cast<size_t>(tokens_per_cta) * (head_dim / 2) * sizeof(float2) +
                      static_cast<size_t>(tokens_per_cta) * sizeof(int32_t);
  if (head_dim == 128) {
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(rope_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    return launch_dependent(rope_kernel<128>, static_cast<unsigned>(grid), kRopeThreads, smem, st, p, tokens_per_cta);
  } else {
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(rope_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    return launch_dependent(rope_kernel<64>, static_cast<unsigned>(grid), kRopeThreads, smem, st, p, tokens_per_cta);
  }
}

// ------------------------------------------------------------ decoder layers
// All windows of a decoder layer in one launch. A CTA takes whole tokens of
// one window (the host gives each window a contiguous range of CTAs). Mode 0
// gathers the window's tokens from the frame-major q, k, v into the packed
// layout the batched attention reads, rotating q and k at window-relative
// (h, w) and absolute frame time; mode 1 writes the window's frames of the
// clean k (rotated) and v into the window's ring slots and its slot table.
// Per token the source row is (f * frame_h + row0 + r) * frame_w + col0 + c;
// every row is H*d contiguous elements, so loads and stores stay coalesced.

namespace {

template <int D, int VPT, bool kThird>
__global__ void __launch_bounds__(kRopeThreads) layer_rope_kernel(const LayerRopeParams p) {
  constexpr int kTarget = kRopeThreads * VPT;   // vectors of each tensor per pass
  constexpr int kPairs = D / 2;
  constexpr int kVecPerHead = D / 8;
  grid_dep_wait();   // the previous kernel of the stream may still be draining
  grid_dep_launch_dependents();
  extern __shared__ float2 smem_layer[];
  const int tpc = p.tokens_per_cta;
  float2* cs_table = smem_layer;                                             // [tpc][D/2]
  int64_t* src_row = reinterpret_cast<int64_t*>(cs_table + tpc * kPairs);   // [tpc]
  int64_t* dst_row = src_row + tpc;                                          // [tpc]
  int32_t* pos = reinterpret_cast<int32_t*>(dst_row + tpc);                  // [tpc][3]: frame, row, column

  // this CTA's window: the last one whose first CTA is not after this CTA
  int wi = 0;
  for (int i = 1; i < p.n_windows; ++i)
    if (p.win[i].cta_begin <= static_cast<int>(blockIdx.x)) wi = i;
  const int row0 = p.win[wi].row0, col0 = p.win[wi].col0, cols = p.win[wi].cols;
  const int T_w = p.win[wi].rows * cols;
  const int64_t n0 = p.win[wi].n_committed;
  const int first = p.win[wi].first_frame;
  const int wf = p.win[wi].window_frames;
  const int tok_lo = (static_cast<int>(blockIdx.x) - p.win[wi].cta_begin) * tpc;
  const int ntok = min(tpc, p.win[wi].n_tok - tok_lo);
  if (ntok <= 0) return;
  const int vpt = p.n_heads * kVecPerHead;   // 16-byte vectors per token
  const int nvec = ntok * vpt;
  const bool commit = p.mode == 1;

  // the window's slot table: frame g = n + f now lives in slot g mod W
  if (commit && tok_lo == 0) {
    int32_t* slots = p.win[wi].slot_frame;
    const int frames = p.win[wi].n_tok / T_w;
    for (int f = threadIdx.x; f < frames; f += kRopeThreads) {
      const int64_t g = n0 + first + f;
      slots[g % wf] = static_cast<int32_t>(g);
    }
  }

  // source row, destination row and (frame, row, column) of every token
  for (int t = threadIdx.x; t < ntok; t += kRopeThreads) {
    const int j = first * T_w + tok_lo + t;   // token of the window's chunk, frame by frame
    const int f = j / T_w;
    const int rc = j - f * T_w;
    const int r = rc / cols;
    const int c = rc - r * cols;
    src_row[t] = (static_cast<int64_t>(f) * p.frame_h + row0 + r) * p.frame_w + col0 + c;
    dst_row[t] = commit ? static_cast<int64_t>((n0 + f) % wf) * T_w + rc : p.win[wi].packed_row0 + j;
    pos[3 * t] = f;
    pos[3 * t + 1] = r;
    pos[3 * t + 2] = c;
  }
  __syncthreads();

  const uint4* s0 = reinterpret_cast<const uint4*>(p.src[0]);
  const uint4* s1 = reinterpret_cast<const uint4*>(p.src[1]);
  const uint4* s2 = reinterpret_cast<const uint4*>(p.src[2]);   // read only when kThird
  uint4* d0 = reinterpret_cast<uint4*>(commit ? p.win[wi].ring_k : p.dst[0]);
  uint4* d1 = reinterpret_cast<uint4*>(commit ? p.win[wi].ring_v : p.dst[1]);
  uint4* d2 = reinterpret_cast<uint4*>(p.dst[2]);

  for (int base = 0; base < nvec; base += kTarget) {
    // loads first: they are in flight while the sin/cos table is built
    uint4 a[VPT], b[VPT], c3[kThird ? VPT : 1];
    {
      int j = base + threadIdx.x;
      int t = j / vpt;
      int r = j - t * vpt;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (j < nvec) {
          const int64_t at = src_row[t] * vpt + r;
          a[k] = s0[at];
          b[k] = s1[at];
          if constexpr (kThird) c3[k] = s2[at];
        }
        j += kRopeThreads;
        r += kRopeThreads;
        while (r >= vpt) {
          r -= vpt;
          ++t;
        }
      }
    }

    if (base == 0) {
      for (int i = threadIdx.x; i < ntok * kPairs; i += kRopeThreads) {
        const int t = i / kPairs;
        const int pr = i - t * kPairs;
        const int ax = p.phase.axis[pr];
        const int64_t ps = ax == 0 ? p.t_clock0 + n0 + pos[3 * t] : pos[3 * t + ax];
        const float ang = rope_angle(p.phase.turn_hi[pr], p.phase.turn_lo[pr], ps, p.phase.rad_hi, p.phase.rad_lo);
        float sn, cs;
        sincosf(ang, &sn, &cs);
        cs_table[i] = make_float2(cs, sn);
      }
      __syncthreads();
    }

    int j = base + threadIdx.x;
    int t = j / vpt;
    int r = j - t * vpt;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      if (j < nvec) {
        const float2* cs = cs_table + t * kPairs + (r & (kVecPerHead - 1)) * 4;
        uint32_t* wa = reinterpret_cast<uint32_t*>(&a[k]);
#pragma unroll
        for (int q = 0; q < 4; ++q) wa[q] = rotate_pair(wa[q], cs[q].x, cs[q].y);
        if (!commit) {   // gather: q and k rotate, v is copied; commit: k rotates, v is copied
          uint32_t* wb = reinterpret_cast<uint32_t*>(&b[k]);
#pragma unroll
          for (int q = 0; q < 4; ++q) wb[q] = rotate_pair(wb[q], cs[q].x, cs[q].y);
        }
        const int64_t at = dst_row[t] * vpt + r;
        d0[at] = a[k];
        d1[at] = b[k];
        if constexpr (kThird) d2[at] = c3[k];
      }
      j += kRopeThreads;
      r += kRopeThreads;
      while (r >= vpt) {
        r -= vpt;
        ++t;
      }
    }
  }
}

size_t layer_smem_bytes(int tpc, int head_dim) {
  return static_cast<size_t>(tpc) * ((head_dim / 2) * sizeof(float2) + 2 * sizeof(int64_t) + 3 * sizeof(int32_t));
}

}  // namespace

// 16-byte vectors of each tensor a thread keeps in flight per pass. Two, in
// both modes: a CTA then holds two tokens of 16 heads x 128, and the many
// short CTAs overlap one another's loads and stores better than fewer, longer
// ones (measured on 720p decoder layers, 7200 tokens: commits of 2, 3, 5, 6, 8
// and 12 vectors took 22.6, 23.0-23.3, 24.7, 24.7, 28.7 and 23.4 us; gathers of
// 2, 3, 4 and 5, 28.4-28.8, 28.7-29.0, 28.8-29.4 and 30.8 us).
constexpr int kLayerVecPerThread = 2;
int layer_vec_per_thread(int) { return kLayerVecPerThread; }

int layer_tokens_per_cta(int n_heads, int head_dim, int mode) {
  return std::max(1, kRopeThreads * layer_vec_per_thread(mode) / (n_heads * head_dim / 8));
}

namespace {
template <int D>
cudaError_t launch_layer_d(const LayerRopeParams& p, int n_ctas, size_t smem, cudaStream_t st) {
  constexpr int V = kLayerVecPerThread;
  auto kernel = p.mode == 1 ? layer_rope_kernel<D, V, false>
                            : (p.src[2] != nullptr ? layer_rope_kernel<D, V, true> : layer_rope_kernel<D, V, false>);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  return launch_dependent(kernel, static_cast<unsigned>(n_ctas), kRopeThreads, smem, st, p);
}
}  // namespace

cudaError_t launch_layer_rope(const LayerRopeParams& p, int head_dim, int n_ctas, cudaStream_t st) {
  if (n_ctas <= 0) return cudaSuccess;
  const size_t smem = layer_smem_bytes(p.tokens_per_cta, head_dim);
  return head_dim == 128 ? launch_layer_d<128>(p, n_ctas, smem, st) : launch_layer_d<64>(p, n_ctas, smem, st);
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
__global__ void zero_words_kernel(int32_t* words, int n) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) words[i] = 0;
}
}  // namespace

// Advance the device frame counter after a commit: its own launch, so that
// every CTA of the commit read the old value.
__global__ void advance_frames_kernel(int64_t* counter, int64_t add) { *counter += add; }

cudaError_t launch_advance_frames(int64_t* counter, int64_t add, cudaStream_t st) {
  return launch_plain(advance_frames_kernel, 1, 1, st, counter, add);
}

cudaError_t launch_copy16(void* dst, const void* src, size_t bytes, cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(bytes / 16);
  if (n == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 152 * 16);
  return launch_plain(copy16_kernel, static_cast<unsigned>(blocks), 256, st, static_cast<uint4*>(dst),
                     static_cast<const uint4*>(src), n);
}

cudaError_t launch_init_ring_state(int32_t* slot_frame, int W, int32_t* err_word, int32_t* ws_ctr, int n_ctr,
                                   cudaStream_t st) {
  return launch_plain(init_ring_state_kernel, 1, 256, st, slot_frame, W, err_word, ws_ctr, n_ctr);
}

cudaError_t launch_zero_words(int32_t* words, int n, cudaStream_t st) {
  return launch_plain(zero_words_kernel, 1, 256, st, words, n);
}

}  // namespace sr
