// sr_kernels.h -- parameter blocks and launchers shared by the host API
// (sr_api.cu) and the kernels. Internal to libsr.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <utility>

#include "sr.h"

namespace sr {

// Launch with programmatic stream serialization: the grid may be scheduled
// while the previous kernel of the stream drains, and waits for it on the
// device (grid_dep_wait) before touching global memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                                    cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Plain launch whose status is the launch's own: the <<<>>> form reports
// failures only through cudaGetLastError, which would also return (and clear)
// an unrelated error the caller left pending.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_plain(void (*kernel)(KArgs...), unsigned grid, unsigned block, cudaStream_t st,
                                Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.stream = st;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ------------------------------------------------------------ attention
// One session's view for one launch: up to four key/value segments -- the sink
// bank of the step, the visible ring frames as one or two contiguous row
// ranges (two when a history window wraps around the end of the ring), and
// the chunk itself -- each a 2D tensor map over [rows][H*d] bf16 with a
// {64, 128} box and 128-byte swizzle. A segment with zero rows has no map and
// contributes no tiles.
constexpr int kSegs = 4;
struct alignas(128) AttnSession {
  CUtensorMap kmap[kSegs];
  CUtensorMap vmap[kSegs];
  int32_t seg_rows[kSegs];
  int32_t q_row0;       // first row of this session in the packed q / o
  int32_t lq;           // query rows
  int32_t nqb;          // query blocks of 256 rows
  int32_t nfull;        // blocks per head run as whole units: all of them, or all but a
                        // single-tile (<= 128-row) last block
  int32_t ntail;        // 1 when the last block is a single tile (run with the last-block units), else 0
  int32_t unit_begin;   // first whole-block unit of this session (whole blocks come first)
  int32_t tail_begin;   // index of this session's last-block units among all last-block units
  float* ws_part;       // key-split partials: [H][kMaxTailSplit][128][d + 4] fp32 (NULL: no split)
  int32_t* ws_ctr;      // [H] per-head arrival counters (epoch << 4 | count)
  int32_t epoch;        // this call's epoch for the counters (increases per call of the session)
  // Device frame counter (NULL: the host filled seg_rows). When set, segments 1
  // and 2 are maps over the whole ring and the kernel derives the visible ring
  // rows from *dev_n: the last hist_req committed frames (-1: every occupied slot).
  const int64_t* dev_n;
  int32_t hist_req;
  int32_t ring_W;
  int32_t ring_T;
};

template <int NSESS>
struct alignas(128) AttnParams {
  CUtensorMap qmap;               // packed q, [total_rows][H*d]
  AttnSession sess[NSESS];
  // Unit ranges of the sessions, packed so that finding a unit's session reads
  // a few contiguous words rather than one field of each (large) session:
  // whole-block units of session i end at whole_end[i], its last-block units
  // (among all last-block units) at tail_end[i].
  int32_t whole_end[NSESS];
  int32_t tail_end[NSESS];
  int32_t n_sess;
  int32_t n_full_units;           // whole 256-row blocks (all sessions); last blocks follow
  int32_t n_conv;                 // the last n_conv whole blocks each run as two single-tile units,
                                  // which balance the end of the launch
  int32_t tail_split;             // key-range parts per single-tile last block (1: no key split)
  int32_t n_heads;
  float scale_log2;               // softmax scale * log2(e)
  int32_t lse_ld;                 // row stride of lse ([H][lse_ld]); 0 when lse is NULL
  __nv_bfloat16* o;               // packed output, [total_rows][H][d]
  float* lse;
  int32_t* err_word;
  uint64_t timeout_ns;
  int32_t n_units;                // work units of the launch
  int32_t epoch;                  // tags the unit counter (the first session's call epoch)
  // Launch-wide unit counter and count of CTAs that ran out of units (two
  // words in the first session's workspace). NULL: one unit per CTA.
  unsigned long long* unit_ctr;
};

constexpr int kAttnThreads = 512;  // 2 softmax warpgroups; MMA warp, TMA warp, 2 idle warps; the epilogue warpgroup
constexpr int kAttnMaxBatch = SR_MAX_BATCH;
// A kernel's parameters may take at most 32764 bytes.
static_assert(sizeof(AttnParams<kAttnMaxBatch>) <= 32764, "attention parameters exceed the kernel parameter limit");

int attn_smem_bytes(int head_dim);
cudaError_t attn_prepare(int head_dim, int nsess_template);   // sets the smem attribute
// Grid: one CTA per unit, or, with a unit counter, one CTA per SM (at most
// one per unit) taking units until none are left.
cudaError_t launch_attention_1(const AttnParams<1>& p, int head_dim, cudaStream_t st);
cudaError_t launch_attention_n(const AttnParams<kAttnMaxBatch>& p, int head_dim, cudaStream_t st);
int sm_count();   // SMs of the current device

// ------------------------------------------------------------ RoPE / commit
// Rotary pairs of a head: pair p (dims 2p, 2p+1) belongs to axis t, h or w and
// turns by c_p = base^(-2i/d_axis) / (2 pi) turns per position step, held as
// the 96-bit binary fraction C_p = round(c_p * 2^96) = turn_hi * 2^32 + turn_lo
// (computed on the host in rope_phase.cu).
constexpr int kMaxPairs = 64;
struct RopePhase {
  uint64_t turn_hi[kMaxPairs];
  uint32_t turn_lo[kMaxPairs];
  int8_t axis[kMaxPairs];      // 0 = t, 1 = h, 2 = w
  float rad_hi, rad_lo;        // 2 pi / 2^32 = rad_hi + rad_lo
};
void rope_phase_table(float base, int head_dim, RopePhase* out);

// Positions whose angle rope_angle forms exactly: |pos| < 2^42 keeps the
// rounding of C_p below 2^-55 turns.
constexpr int64_t kRopePositionLimit = int64_t(1) << 42;

// The angle, in radians reduced into [-pi, pi), of a pair with turn constant
// (hi, lo) at integer position pos, |pos| < kRopePositionLimit. The phase
// frac(pos * C / 2^96), in units of 2^-64 turn, is formed with 64-bit integer
// arithmetic (wrapping modulo 2^64 drops whole turns and nothing else), read
// as a signed turn in [-1/2, 1/2) and scaled by 2 pi in two float parts. The
// host and the kernels run this same function; every float operation is
// exact or an explicit fmaf, so both get the same bits.
__host__ __device__ inline float rope_angle(uint64_t hi, uint32_t lo, int64_t pos, float rad_hi, float rad_lo) {
  const uint64_t a = pos < 0 ? 0ull - static_cast<uint64_t>(pos) : static_cast<uint64_t>(pos);
  // floor(a * C / 2^32) mod 2^64 = a * hi + floor(a * lo / 2^32)
  uint64_t ph = a * hi + (a >> 32) * lo + (((a & 0xffffffffull) * lo) >> 32);
  if (pos < 0) ph = 0ull - ph;   // frac(-x) = -frac(x) modulo one turn
  const int64_t s = static_cast<int64_t>(ph);
  const int32_t w = static_cast<int32_t>(s >> 32);   // turns in units of 2^-32
  const float f_hi = static_cast<float>(w);          // rounded; the rest goes to f_lo
  const float f_lo = fmaf(static_cast<float>(static_cast<uint32_t>(s)), 0x1p-32f,
                          static_cast<float>(static_cast<int64_t>(w) - static_cast<int64_t>(f_hi)));
  return fmaf(f_hi, rad_hi, fmaf(f_hi, rad_lo, f_lo * rad_hi));
}

struct RopeParams {
  RopePhase phase;
  const __nv_bfloat16* src0;   // rotated
  const __nv_bfloat16* src1;   // rotated (mode 0) or copied (mode 1)
  __nv_bfloat16* dst0;
  __nv_bfloat16* dst1;
  int32_t* slot_frame;         // mode 1 only
  int64_t n_committed;         // frames committed before this chunk
  int32_t n_tok;               // F*T
  int32_t n_heads;
  int32_t tokens_per_frame;    // T
  int32_t grid_w;
  int32_t window_frames;       // W (mode 1)
  int32_t chunk_frames;        // F (mode 1)
  int32_t t_clock0;
  int32_t mode;                // 0: rotate src0->dst0 and src1->dst1 in place; 1: commit
  const int64_t* dev_n;        // device frame counter: when set, frame f's time and slot use
                               // *dev_n + n_committed + f (n_committed is then an offset)
};

cudaError_t launch_rope(const RopeParams& p, int head_dim, cudaStream_t st);

// A decoder layer's windows in one launch: gather from frame-major tensors
// [F][frame_h][frame_w][H][d] into the window-packed layout with RoPE at
// window-relative (h, w) (mode 0), or write every window's ring slots (mode 1).
constexpr int kMaxLayerWindows = SR_MAX_LAYER_WINDOWS;
struct LayerWindow {
  int32_t row0, col0, rows, cols;   // the window in the frame
  int64_t packed_row0;              // mode 0: first packed row of the window
  int64_t n_committed;              // frames the window's session committed before this chunk
  __nv_bfloat16* ring_k;            // mode 1: the window's ring [W*rows*cols][H][d]
  __nv_bfloat16* ring_v;
  int32_t* slot_frame;              // mode 1: [W]
  int32_t window_frames;            // mode 1: W
  int32_t first_frame;              // first chunk frame processed (mode 1: F - W when F > W, else 0)
  int32_t cta_begin;                // first CTA of this window
  int32_t n_tok;                    // tokens processed
};
struct LayerRopeParams {
  RopePhase phase;
  const __nv_bfloat16* src[3];      // frame-major: q, k, v (mode 0) or k_raw, v (mode 1); v may be NULL in mode 0
  __nv_bfloat16* dst[3];            // mode 0: packed q, k, v
  int32_t frame_h, frame_w;
  int32_t n_heads;
  int32_t t_clock0;
  int32_t mode;                     // 0: gather + rotate q, k (+ copy v); 1: commit k (rotated) and v
  int32_t n_windows;
  int32_t tokens_per_cta;
  LayerWindow win[kMaxLayerWindows];
};
cudaError_t launch_layer_rope(const LayerRopeParams& p, int head_dim, int n_ctas, cudaStream_t st);
int layer_tokens_per_cta(int n_heads, int head_dim, int mode);

// ------------------------------------------------------------ misc
cudaError_t launch_copy16(void* dst, const void* src, size_t bytes, cudaStream_t st);
cudaError_t launch_init_ring_state(int32_t* slot_frame, int W, int32_t* err_word, int32_t* ws_ctr, int n_ctr,
                                   cudaStream_t st);
cudaError_t launch_advance_frames(int64_t* counter, int64_t add, cudaStream_t st);
cudaError_t launch_zero_words(int32_t* words, int n, cudaStream_t st);

constexpr int kMaxTailSplit = SR_MAX_TAIL_SPLIT;

// Used only by the allocation-free entry point (sr_noalloc.cu): validate a
// chunk-attention call against a scratch area of scratch_bytes (no side
// effects), then launch it with that scratch standing in for the session's
// workspace. Neither allocates anything.
sr_status attention_scratch_check(const sr_session* s, int32_t step, const void* q, const void* k, const void* v,
                                  const void* o, const float* lse, uint64_t scratch_bytes);
sr_status attention_into_scratch(sr_session* s, int32_t step, const void* q, const void* k, const void* v, void* o,
                                 float* lse, void* stream, void* scratch);
int session_heads(const sr_session* s);
// workspace layout: the launch-wide unit counter (two 64-bit words), the
// per-head arrival counters (together padded to 256 B), then the partials
constexpr size_t kWsUnitCtrBytes = 16;
inline size_t ws_counter_bytes(int n_heads) {
  return (kWsUnitCtrBytes + static_cast<size_t>(n_heads) * 4 + 255) / 256 * 256;
}
inline size_t ws_partial_floats_per_head(int head_dim) { return static_cast<size_t>(kMaxTailSplit) * 128 * (head_dim + 4); }
cudaError_t launch_debug_wait(int32_t* err_word, uint64_t timeout_ns, cudaStream_t st);

}  // namespace sr
