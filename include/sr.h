/*
 * sr.h -- C ABI of the streaming chunk-attention library (libsr.so), GB300 / sm_103a.
 *
 * The operations follow the streaming loop of the StreamRender-H3 project page
 * ("Interactive Coding Worlds with Real-time Streaming Diffusion Render", NVlabs
 * Sol-Engine), cited below as [H3 page]:
 *   - condition once per session: the static context (sink) keys/values exist
 *     once per denoising step, for the whole session, and every chunk reads them
 *     ([H3 page] section 3.3 "Static-context KV caching");
 *   - two denoising steps per chunk ([H3 page] 3.1.3 "Two-step generation"), each
 *     attending bidirectionally over sink + recent history + the chunk itself
 *     ([H3 page] 3.1.2);
 *   - after the last step the chunk's keys receive their rotary position once and
 *     are written in place into a preallocated ring buffer, evicting the oldest
 *     frames ([H3 page] 3.2 Iteration 3 item 2; 3.3 "Persistent KV layout").
 *
 * Conventions shared by every call
 *   - Tensors are bf16, token-major [L][H][d], contiguous: row stride H*d elements.
 *     Every device pointer must be 16-byte aligned.
 *   - All calls are asynchronous on the given stream (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream) and enqueue in call order. The
 *     RoPE/commit and attention kernels launch with programmatic stream
 *     serialization: their CTAs may be scheduled while the previous kernel of
 *     the stream drains, but they touch no global memory before it has
 *     completed, so stream order holds for every buffer.
 *   - The library never allocates or frees device memory and never synchronises
 *     a stream: every device buffer is owned by the caller and must outlive the
 *     session; they are kept in the layout the attention kernel loads, so nothing
 *     is repacked between calls ([H3 page] 3.3 "Persistent KV layout"). The only
 *     host allocation is the session handle.
 *   - Arguments are validated before anything is launched; a rejected call
 *     changes no state. A failed launch returns SR_ERR_CUDA.
 *   - Device-side waits are bounded. A wait that runs out of time writes a
 *     nonzero code into the caller's err_word (first error wins) and the kernel
 *     returns; the caller reads err_word after synchronising and may map it with
 *     sr_device_error_status().
 *   - A session is not thread-safe; distinct sessions are independent.
 */
#ifndef SR_H_
#define SR_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SR_API __attribute__((visibility("default")))
#else
#define SR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct sr_session sr_session;   /* opaque host handle */

typedef enum {
  SR_OK = 0,
  SR_ERR_INVALID_ARG = -1,   /* NULL pointer, bad size, step out of range, ... */
  SR_ERR_UNSUPPORTED = -2,   /* e.g. head_dim other than 64 or 128 */
  SR_ERR_ALIGN = -3,         /* a device pointer is not 16-byte aligned */
  SR_ERR_STATE = -4,         /* call not allowed in the session's current state */
  SR_ERR_CUDA = -5,          /* a CUDA runtime/driver call or a launch failed */
  SR_ERR_TIMEOUT = -6        /* a device wait ran out of time (from err_word) */
} sr_status;

/* Device error codes written into err_word (0 = no error). */
enum {
  SR_DEVERR_NONE = 0,
  SR_DEVERR_WAIT_TIMEOUT = 1  /* low 8 bits; bits 8..15 name the wait site */
};

/* Session shape and constants. */
typedef struct {
  int32_t n_heads;          /* H >= 1 */
  int32_t head_dim;         /* d: 64 or 128 */
  int32_t grid_h, grid_w;   /* latent grid; T = grid_h*grid_w tokens per frame, row-major (h, w) */
  int32_t chunk_frames;     /* F >= 1 latent frames per chunk; Lq = F*T queries */
  int32_t window_frames;    /* W: ring capacity in frames; 0 (no history) or >= F */
  int32_t n_sink;           /* S >= 0 sink tokens per denoising step */
  int32_t n_steps;          /* number of denoising steps = number of sink banks, >= 1 */
  int32_t t_clock0;         /* rotary time position of stream frame 0 */
  float rope_base;          /* rotary base (e.g. 10000); > 1 */
  float softmax_scale;      /* <= 0 selects 1/sqrt(head_dim) */
  uint64_t wait_timeout_ns; /* bound on every device-side wait; 0 selects 2 s */
  int32_t tail_split;       /* key-range split of a chunk's last, single-tile query block into
                               work units: 0 = chosen per call, 1 = never, 2..4 = exactly that many
                               (needs a workspace; clamped to the number of key tiles) */
} sr_config;

/* Caller-owned device buffers of one session (all 16-byte aligned). */
typedef struct {
  void* sink_k;             /* [n_steps][S][H][d] bf16: static context bank, final (no RoPE applied by the library) */
  void* sink_v;             /* [n_steps][S][H][d] bf16 */
  void* ring_k;             /* [W*T][H][d] bf16: rotated keys of committed frames, slot s = rows [s*T, (s+1)*T) */
  void* ring_v;             /* [W*T][H][d] bf16 */
  int32_t* slot_frame;      /* [W] int32: absolute frame held by each slot, -1 = empty */
  int32_t* err_word;        /* [1] int32: device error word (see SR_DEVERR_*) */
  void* workspace;          /* optional, 256-byte aligned, sr_workspace_bytes() long: the work
                               counter of persistent attention launches and the partial results of
                               key-split last blocks. NULL: one CTA per work unit and no split. The
                               library initialises it in sr_session_init; do not modify it after. */
  int64_t* frame_counter;   /* optional [1] int64 device: the committed-frame count the *_dev calls
                               read and advance on the device (NULL: those calls are refused).
                               When given, sr_session_init zeroes it and zero-fills ring_k/ring_v. */
} sr_buffers;

#define SR_MAX_TAIL_SPLIT 4

/*
 * Bytes of workspace a session with this config can use (see sr_buffers.workspace):
 * a launch-wide work counter, and per head a counter and SR_MAX_TAIL_SPLIT partial
 * results of 128 rows.
 */
SR_API sr_status sr_workspace_bytes(const sr_config* cfg, uint64_t* bytes);

/*
 * The plan sr_chunk_attention uses for one query group (host arithmetic only; no
 * device is needed when sm_count > 0): lq query rows over key_tiles 128-row key
 * tiles, n_heads heads. The launch runs whole 256-row blocks first, then the
 * single-tile last blocks (lq mod 256 in 1..128), each split into *parts key-range
 * parts (needs a workspace; tail_split > 0 forces the count, clamped to 1..key_tiles
 * and SR_MAX_TAIL_SPLIT). *whole_as_tiles of the last whole blocks run as two
 * single-tile units each, to balance a partly filled last wave of sm_count SMs
 * (<= 0: the current device's). The choice comes from simulating the dispatch of
 * the units, longest first, to the SM that frees up first. *n_units: units of the
 * launch. SR_ERR_INVALID_ARG for NULL outputs or sizes out of range.
 */
SR_API sr_status sr_plan_attention(int32_t n_heads, int64_t lq, int64_t key_tiles, int32_t has_workspace,
                                   int32_t tail_split, int32_t sm_count, int32_t* parts, int32_t* whole_as_tiles,
                                   int64_t* n_units);

/*
 * Create a session. Copies the sink banks from sink_k_src / sink_v_src (device,
 * same layout as the bank) into bufs->sink_k / sink_v when they are non-NULL
 * (NULL: the bank already holds them), fills slot_frame with -1, clears
 * err_word and sets the committed-frame count n to 0. The static context is
 * written once ([H3 page] 3.3 "Static-context KV caching", "Persistent KV layout").
 * On success *out receives the handle; on failure *out is left NULL.
 */
SR_API sr_status sr_session_init(const sr_config* cfg, const sr_buffers* bufs,
                          const void* sink_k_src, const void* sink_v_src,
                          void* stream, sr_session** out);

/*
 * Declare that the caller has put the ring into the state reached after
 * n_committed frames (checkpoint / resume, or a synthetic mid-stream start):
 * frame g in slot g mod W for the last min(n_committed, W) frames, and
 * slot_frame filled accordingly. Only the host mirror of n changes.
 * 0 <= n_committed <= 2^31 - 1 (slot_frame holds frame indices as int32), else
 * SR_ERR_INVALID_ARG.
 */
SR_API sr_status sr_session_restore(sr_session* s, int64_t n_committed);

/* Frames committed so far (host mirror of the ring state). */
SR_API sr_status sr_session_frames(const sr_session* s, int64_t* n_committed);

/*
 * In-place 3D (t, h, w) rotary positions on the chunk's queries and keys
 * ([H3 page] 3.2 Iteration 3 item 2 and Iteration 4: absolute latent-frame
 * time, so that a score is a function of the time gap only).
 * q, k: [F*T][H][d] bf16, rotated in place. Token n lies in frame f = n / T,
 * row (n % T) / grid_w, column n % grid_w; its time is t_clock0 + n_committed + f.
 * The head dim splits into [d_t | d_h | d_w], d_h = d_w = 2*floor(d/6); inside an
 * axis, pair (x[2i], x[2i+1]) turns by p * rope_base^(-2i/d_axis). The angle is
 * reduced modulo 2*pi exactly, whatever the stream time (see sr_rope_angle); the
 * rotation is computed in fp32 and stored bf16 round-to-nearest-even. Either
 * pointer may be NULL to skip it.
 */
SR_API sr_status sr_rope3d_qk(sr_session* s, void* q, void* k, void* stream);

/*
 * Attention of the chunk's queries for denoising step `step`
 * ([H3 page] 3.1.2: bidirectional inside the window; "Prefix cache": the moving
 * rows see every key of the window; 3.3: each step reads its own bank):
 *   O = softmax(scale * Q K^T) V  over  sink bank[step] U occupied ring slots U chunk.
 * q, k, v: [F*T][H][d] bf16 (q and k already rotated); o: [F*T][H][d] bf16 output.
 * lse: optional [H][F*T] fp32 natural-log sum-exp of the scaled scores (NULL to skip).
 * bf16 operands, fp32 accumulation and fp32 online softmax on the tensor cores.
 * When the chunk's last 256-row query block holds a single 128-row tile and the
 * session has a workspace, that block's key range may be split over several work units
 * (sr_config.tail_split); the last part to finish merges the partial results. With a
 * workspace the launch is persistent (one CTA per SM taking work units from a counter
 * in the workspace). Calls of one session that overlap on the GPU race on that
 * workspace. After a device timeout (err_word set) initialise the session again: a
 * CUDA-graph replay of the same launch could otherwise inherit a stale count.
 */
SR_API sr_status sr_chunk_attention(sr_session* s, int32_t step, const void* q, const void* k,
                             const void* v, void* o, float* lse, void* stream);

/*
 * Commit the clean chunk after the last denoising step ([H3 page] 3.2 Iteration 3
 * item 2: the rotary position is applied a single time, at the store into the
 * frame's fixed slot; 3.3 "Persistent KV layout": the cache is modified where it
 * lives). k_raw (un-rotated) and v:
 * [F*T][H][d] bf16. Frame g = n + f goes to slot g mod W with its keys rotated at
 * time t_clock0 + g; slot_frame[g mod W] = g; then n += F. The frames previously
 * held by those slots are evicted. With W = 0 only n advances. A session commits
 * at most 2^31 - 1 frames (slot_frame is int32): a commit past that returns
 * SR_ERR_STATE and changes nothing.
 */
SR_API sr_status sr_cache_commit(sr_session* s, const void* k_raw, const void* v, void* stream);

/* Free the host handle (device buffers stay the caller's). NULL is accepted. */
SR_API sr_status sr_session_free(sr_session* s);

/*
 * One launch for several sessions' chunks (multi-session serving; the page's
 * per-request cache banks and reused attention metadata, [H3 page] 3.3).
 * sessions[0..n-1] must share n_heads, head_dim and softmax scale. q, k, v, o are
 * packed along L: session i owns rows [q_off[i], q_off[i+1]) (q_off is a HOST
 * array of n+1 offsets, q_off[0] = 0, q_off[i+1]-q_off[i] = that session's F*T).
 * Each session attends over its own bank[step], its own ring and its own rows.
 * lse (optional) is [H][q_off[n]] fp32. 1 <= n <= SR_MAX_BATCH.
 */
#define SR_MAX_BATCH 24
SR_API sr_status sr_chunk_attention_batch(sr_session* const* sessions, int32_t n, int32_t step,
                                   const void* q, const void* k, const void* v,
                                   const int64_t* q_off, void* o, float* lse, void* stream);

/*
 * sr_chunk_attention for callers that cannot allocate device memory. (The pages
 * have no counterpart: this is a deployment convenience of this library.)
 * Some callers cannot call cudaMalloc or hand over a workspace: code running inside
 * a framework's fixed memory pool, a plugin that must not touch the allocator, or a
 * process that only receives a stream and its tensors. This entry point computes
 * exactly what sr_chunk_attention computes, with the same arguments, but the scratch
 * of key-split last blocks comes from a 16 MiB array compiled into the library
 * (held on every GPU that loads it until the process exits) instead of the
 * session's workspace, which may be NULL. It allocates nothing.
 * - Limit: sessions whose sr_workspace_bytes() exceeds 16 MiB (for example more
 *   than 62 heads at head_dim 128) are rejected with SR_ERR_UNSUPPORTED before
 *   anything is launched.
 * - The first call on a device does one-time set-up (it looks up the array's device
 *   address and sets the kernel's shared-memory limit); make that first call before
 *   any stream capture.
 * - Every call shares the one array: the counters that must start at zero are
 *   cleared on the stream before each launch, and calls that overlap on the GPU
 *   (other streams, other threads, other sessions) race on it.
 */
SR_API sr_status sr_chunk_attention_noalloc(sr_session* s, int32_t step, const void* q, const void* k,
                                            const void* v, void* o, float* lse, void* stream);

/*
 * The pages' unit rhythm ([teardown] "A window that slides, and a prefix that
 * doesn't"; [H3 page] 3.1.2). The video codec turns 17 RGB frames into 5 latent
 * frames, the first of every five covering one RGB frame; with single-frame latents
 * merged into their neighbour, scheduling units hold 2, 1, 1, 1 latents and repeat.
 * A stream opens with one window of bootstrap_units units, then every chunk is
 * chunk_units units and sees the window_units units right before it as recent
 * history; the sink is the first sink_units units. With the shipped values (7, 2,
 * 2, 2, merged) the first window is 9 latents and the chunks alternate 3 and 2
 * latents with 2 and 3 latents of history.
 * Host-only arithmetic (no GPU call): fills *out for chunk `chunk_index` (0 = the
 * first window, which has no history). Invalid (non-positive unit counts, negative
 * index, sums past int32): SR_ERR_INVALID_ARG.
 */
typedef struct {
  int32_t first_frame;   /* stream index of the chunk's first latent frame */
  int32_t n_frames;      /* latent frames in the chunk */
  int32_t hist_frames;   /* latent frames of recent history the chunk sees */
  int32_t sink_frames;   /* latent frames in the sink units */
} sr_chunk_plan;
SR_API sr_status sr_plan_chunk(int32_t chunk_index, int32_t bootstrap_units, int32_t chunk_units,
                               int32_t window_units, int32_t sink_units, int32_t merge_single_frame_units,
                               sr_chunk_plan* out);

/*
 * The per-chunk calls for chunks of any length (the unit rhythm above).
 * n_frames: latent frames in this chunk, 1 <= n_frames and n_frames*T*H*d within the
 * limits sr_session_init applies to chunk_frames (sr_config.chunk_frames is the
 * length the plain calls use). q, k, v, o, k_raw: [n_frames*T][H][d] bf16.
 * - sr_rope3d_qk_frames: as sr_rope3d_qk, frames n .. n+n_frames-1.
 * - sr_chunk_attention_frames: as sr_chunk_attention over sink bank[step] U the last
 *   hist_frames committed frames U the chunk; hist_frames = -1 means every occupied
 *   slot (what sr_chunk_attention sees), otherwise 0 <= hist_frames <= min(n, W).
 *   The visible frames may wrap around the end of the ring. lse: [H][n_frames*T].
 * - sr_cache_commit_frames: as sr_cache_commit for n_frames frames, which may wrap
 *   around the end of the ring; when n_frames > W only the chunk's last W frames
 *   are written (its earlier frames would be evicted by its later ones), and n
 *   still advances by n_frames.
 */
SR_API sr_status sr_rope3d_qk_frames(sr_session* s, int32_t n_frames, void* q, void* k, void* stream);
SR_API sr_status sr_chunk_attention_frames(sr_session* s, int32_t step, int32_t n_frames, int32_t hist_frames,
                                           const void* q, const void* k, const void* v, void* o, float* lse,
                                           void* stream);
SR_API sr_status sr_cache_commit_frames(sr_session* s, int32_t n_frames, const void* k_raw, const void* v,
                                        void* stream);

/*
 * The page-faithful window ([teardown] "A window that slides, and a prefix that
 * doesn't"; [H3 page] 3.1.2 "Prefix cache"). The pages split each window into a
 * fixed prefix (conditioning and sink, whose keys and values are the per-step bank)
 * and a moving part (recent history and the chunk, recomputed every chunk), with an
 * asymmetric mask: prefix rows attend only to the prefix, moving rows attend to the
 * whole window. One launch computes both groups; the mask is expressed as each
 * group's key set, so no score is masked:
 *   prefix rows:  softmax(scale Q_p K_bank^T) V_bank
 *   moving rows:  softmax(scale Q_m [K_bank; K_m]^T) [V_bank; V_m]
 * moving_frames: latent frames of moving rows (history + chunk), M = moving_frames*T.
 * q, o: [P + M][H][d] bf16 with P = n_sink when with_prefix != 0 (the prefix rows
 * first, as the prefix pass of a session's first window), else P = 0.
 * k_moving, v_moving: [M][H][d] bf16, the moving rows' keys and values (not the
 * ring: this is the computation the ring path caches). lse: optional [H][P + M].
 * with_prefix needs n_sink > 0. The ring and the frame count are not touched.
 */
SR_API sr_status sr_window_attention(sr_session* s, int32_t step, int32_t moving_frames, int32_t with_prefix,
                                     const void* q, const void* k_moving, const void* v_moving, void* o,
                                     float* lse, void* stream);

/*
 * sr_rope3d_qk for rows of n_frames frames starting at the stream's frame
 * first_frame (time t_clock0 + first_frame + f): recomputed history rows keep their
 * own frame times. |first_frame| <= 2^40, else SR_ERR_INVALID_ARG.
 */
SR_API sr_status sr_rope3d_qk_at(sr_session* s, int64_t first_frame, int32_t n_frames, void* q, void* k,
                                 void* stream);

/*
 * Device-resident chunk state, for CUDA-graph capture of the per-chunk sequence
 * ([H3 page] 3.3 "Attention metadata reuse": the per-call metadata is prepared once
 * and no call waits on the host). These calls compute exactly what sr_rope3d_qk_frames,
 * sr_chunk_attention_frames and sr_cache_commit_frames compute, but the
 * committed-frame count n is read from bufs->frame_counter when the kernels run, and
 * sr_cache_commit_dev advances it on the device (one more tiny launch). One captured
 * sequence of these calls therefore serves every chunk of its length:
 *   capture:  rope_dev(step 0), attention_dev(0), rope_dev(1), attention_dev(1), commit_dev
 *   replay:   once per chunk, after copying the chunk's inputs into the captured buffers.
 * The visible ring rows come from the counter (hist_frames as in
 * sr_chunk_attention_frames, -1 = every occupied slot, otherwise at most W; fewer
 * frames are seen while fewer are committed). Ring tiles that straddle the end of the
 * visible rows read neighbouring ring rows with zero weight, so the ring must hold
 * finite values: sr_session_init zero-fills it when a frame_counter is given.
 * The host mirror of n (sr_session_frames) does not follow replays; sr_session_restore
 * re-synchronises it before host-state calls are mixed in.
 * The frame-count limit of the host-state calls (2^31 - 1 committed frames, the
 * int32 slot table) holds here too, but the host cannot see replays: the caller
 * keeps a replayed session below it. Without a frame_counter: SR_ERR_STATE.
 */
SR_API sr_status sr_rope3d_qk_dev(sr_session* s, int32_t n_frames, void* q, void* k, void* stream);
SR_API sr_status sr_chunk_attention_dev(sr_session* s, int32_t step, int32_t n_frames, int32_t hist_frames,
                                        const void* q, const void* k, const void* v, void* o, float* lse,
                                        void* stream);
SR_API sr_status sr_cache_commit_dev(sr_session* s, int32_t n_frames, const void* k_raw, const void* v,
                                     void* stream);

/*
 * Window partition of the pages' streaming decoder ([H3 page] 3.2 Iteration 2
 * "Space": attention within non-overlapping windows of window x window tokens, every
 * other layer shifted by half a window; Iteration 3 item 4: each window is one short
 * variable-length sequence, padding positions left out). Host-only arithmetic.
 * A frame of grid_h x grid_w tokens is cut at rows/columns shift - window, shift,
 * shift + window, ... (shift = 0 for the plain layers, window / 2 for the shifted ones)
 * and clipped to the frame, so edge windows are smaller. Windows are numbered row
 * by row. sr_window_count gives their number; sr_plan_window fills *out for window
 * `index` (its first token row and column and its size). Each window then attends,
 * per head, over the global tokens U its cached frames U its chunk frames: with this
 * library, one session per window (grid = the window's size, the global tokens as a
 * shared bank), batched by sr_chunk_attention_batch.
 */
typedef struct {
  int32_t row0, col0;      /* first token row and column of the window in the frame */
  int32_t rows, cols;      /* its size (clipped at the frame edges) */
} sr_window;
SR_API sr_status sr_window_count(int32_t grid_h, int32_t grid_w, int32_t window, int32_t shifted, int32_t* count);
SR_API sr_status sr_plan_window(int32_t grid_h, int32_t grid_w, int32_t window, int32_t shifted, int32_t index,
                                sr_window* out);

/*
 * The rotation angle the RoPE and commit kernels apply, as host arithmetic (no
 * GPU call): rotary pair `pair` (0 <= pair < head_dim/2, numbered across
 * [d_t | d_h | d_w]) of a token at integer position `position` on that pair's
 * axis turns by theta = position * rope_base^(-2i/d_axis) ([H3 page] 3.2
 * Iteration 4: the time position is the absolute latent-frame index of the
 * stream, which grows without bound). *angle receives theta reduced into
 * [-pi, pi), rounded to float. The reduction is exact: each pair's
 * rope_base^(-2i/d_axis) / (2*pi) is held as a 96-bit binary fraction, and the
 * phase position * that fraction modulo 1 is formed in integer arithmetic, so
 * the angle is within about 2^-24 rad of the exact reduced value for every
 * |position| < 2^42 (every position the other calls can produce). The kernels run
 * the same arithmetic and then take the fp32 sine and cosine of *angle.
 * SR_ERR_INVALID_ARG for a bad config, pair or position.
 */
SR_API sr_status sr_rope_angle(const sr_config* cfg, int32_t pair, int64_t position, float* angle);

/*
 * A decoder layer's rotary positions, window gather and cache writes, one launch each
 * ([H3 page] 3.2 Iteration 3: the window gather is fused with the rotary embedding;
 * Iteration 6: rotary positions and the K/V cache write in one kernel; Iteration 2
 * "Space": positions relative to the window).
 * sessions[i] is the session of window windows[i] of a frame_h x frame_w latent frame
 * (its grid must be windows[i].rows x windows[i].cols, e.g. from sr_plan_window); all
 * sessions share n_heads, head_dim, chunk_frames F, t_clock0 and rope_base.
 * 1 <= n <= SR_MAX_LAYER_WINDOWS. Frame-major tensors are [F][frame_h][frame_w][H][d]
 * bf16; packed tensors hold the windows' rows back to back in the order of `sessions`
 * (window i from row sum_{j<i} F*rows_j*cols_j; inside a window frame by frame,
 * row-major), the layout sr_chunk_attention_batch reads.
 * - sr_layer_rope_gather: q, k (frame-major) rotated at each window's frames n .. n+F-1
 *   (time t_clock0 + n + f) and window-relative (h, w), written to q_packed, k_packed;
 *   v (optional, NULL to skip) copied to v_packed. The frame-major inputs are not changed.
 * - sr_layer_commit: as sr_cache_commit for every session at once: each window's frames
 *   of k_raw (rotated as above) and v written into its ring slots, its slot table updated,
 *   its n advanced by F.
 * The packed outputs must not overlap the frame-major inputs (every window reads
 * rows of the whole frame while others write), nor one another.
 * Validation failures (SR_ERR_INVALID_ARG, SR_ERR_ALIGN, SR_ERR_STATE as for the
 * per-session calls) change nothing. Calls that overlap on the GPU with other calls
 * of the same sessions race on their rings, as for the per-session calls.
 */
#define SR_MAX_LAYER_WINDOWS 96
SR_API sr_status sr_layer_rope_gather(sr_session* const* sessions, const sr_window* windows, int32_t n,
                                      int32_t frame_h, int32_t frame_w, const void* q, const void* k,
                                      const void* v, void* q_packed, void* k_packed, void* v_packed, void* stream);
SR_API sr_status sr_layer_commit(sr_session* const* sessions, const sr_window* windows, int32_t n,
                                 int32_t frame_h, int32_t frame_w, const void* k_raw, const void* v, void* stream);

/* Map a value read from err_word to SR_OK or SR_ERR_TIMEOUT. */
SR_API sr_status sr_device_error_status(int32_t err_word_value);

/*
 * Diagnostic for the bounded-wait path: launches one block that waits on a
 * barrier nothing will ever complete, using the same bounded wait as the
 * kernels. After timeout_ns it writes SR_DEVERR_WAIT_TIMEOUT (site 0xFF) into
 * *err_word (device, int32) and returns; no copy or tensor-core operation is in
 * flight. Used to test failure detection without faulting or hanging a GPU.
 */
SR_API sr_status sr_debug_wait_timeout(int32_t* err_word, uint64_t timeout_ns, void* stream);

/* Static string for a status code. */
SR_API const char* sr_status_string(sr_status st);

#ifdef __cplusplus
}
#endif
#endif /* SR_H_ */
