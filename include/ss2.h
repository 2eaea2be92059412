/*
 * ss2.h — C ABI of libss2, per-frame SSIMULACRA2 scoring of reference /
 * distorted YUV frame pairs on an NVIDIA GB300 (sm_103a).
 *
 * The operation is the device-resident ssimulacra2 pipeline of
 * "Research-1363: Device-resident ssimulacra2 and a single-wait MS-SSIM on
 * SYCL" (vmafx documentation): section "Sources" lists its steps
 * (picture_to_linear_rgb, linear_rgb_to_xyb, fast_gaussian_1d / blur_plane,
 * multiply_3plane, ssim_map, edge_diff_map, downsample_2x2, pool_score);
 * Findings 2-4 fix the numerics (bit-exact fp32 pipeline up to the sums,
 * double-float per-pixel terms, six 1-norm / 4-norm sums per channel and
 * scale in a fixed reduction tree); the Question asks for the frame to stay
 * on the device with a single read-back.
 *
 * Error convention (errno-style negatives, as the pages' extractors use:
 * "ADR-1357: Run the SYCL CAMBI extractor entirely on the device", Decision,
 * -EINVAL; "ADR-1405: float_ssim_hip decimates on the device ...",
 * Decision 4, -ENOTSUP):
 *   SS2_OK        0
 *   SS2_EINVAL  -22  bad argument; nothing was enqueued
 *   SS2_ENOMEM  -12  device or pinned allocation failed
 *   SS2_ENOTSUP -95  no sm_103 device, or the library was built without one
 *   SS2_EIO      -5  a CUDA runtime call failed; the message is kept
 * The code and message of the last failure on the calling thread are
 * available from ss2_last_error() / ss2_last_error_string().
 *
 * Frame layout: planar Y (width x height), then U, then V (cw x ch each,
 * cw = ceil(width / 2^sx), ch = ceil(height / 2^sy); 4:2:0 sx = sy = 1,
 * 4:2:2 sx = 1, sy = 0, 4:4:4 none), no padding.  8-bit samples are uint8;
 * 9..16-bit samples are little-endian uint16, low-justified.  A call's
 * frames are contiguous: frame f starts at f * ss2_frame_bytes(ctx).
 *
 * Threading: a context is not thread-safe; separate contexts are
 * independent.  Geometry is fixed per context.
 */
#ifndef SS2_H
#define SS2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SS2_OK 0
#define SS2_EINVAL (-22)
#define SS2_ENOMEM (-12)
#define SS2_ENOTSUP (-95)
#define SS2_EIO (-5)

#define SS2_CHROMA_420 420
#define SS2_CHROMA_422 422
#define SS2_CHROMA_444 444

#define SS2_NVALUES 108   /* 3 channels x 6 scales x 2 norms x 3 maps */
#define SS2_NPARAMS 133   /* length of the parameter vector           */
#define SS2_MAX_DIM 16384 /* largest accepted width or height          */

typedef struct ss2_ctx ss2_ctx;

/*
 * ss2_create — a scoring context for one frame geometry on the current
 * CUDA device.  width, height >= 8 and <= SS2_MAX_DIM; bitdepth 8..16;
 * chroma one of 420, 422, 444; subsampled chroma needs an even width
 * (Research-1363, "Sources": the CLI rejects odd widths for 4:2:0).
 * The context owns two device workspaces, each for a batch of frames
 * (chosen from the geometry; ss2_create_batch sets it), used in turn on two
 * internal streams so that consecutive batches overlap on the GPU, and holds
 * the default parameter vector (see ss2_default_params).
 * Returns NULL on failure: -EINVAL (bad geometry), -ENOTSUP (no sm_103
 * device), -ENOMEM, -EIO.
 */
ss2_ctx *ss2_create(int width, int height, int bitdepth, int chroma);

/* ss2_create_batch — as ss2_create with an explicit batch size
 * (1..1024 frames processed per pass over the pipeline).               */
ss2_ctx *ss2_create_batch(int width, int height, int bitdepth, int chroma,
                          int max_batch);

/* ss2_destroy — frees the context and its workspace.  NULL-safe.  Waits for
 * no stream: the caller must not destroy a context with work in flight.  */
void ss2_destroy(ss2_ctx *ctx);

/*
 * ss2_score_frames — scores n_frames frame pairs.
 *   ref, dis: DEVICE pointers, caller-owned, n_frames packed frames each,
 *             read only during the call, not retained.
 *   scores:   HOST array of n_frames doubles, caller-owned.
 *   stream:   cudaStream_t (NULL = legacy default stream); the work starts
 *             after what is already queued on it (the context's two
 *             internal streams wait on an event recorded there, and the
 *             stream waits for them at the end); the call returns after the
 *             scores have reached host memory (one stream synchronisation
 *             per call, 8 bytes read back per frame).
 * n_frames == 0 is a no-op returning 0.  Returns 0 or a negative code;
 * on -EINVAL nothing was enqueued.
 */
int ss2_score_frames(ss2_ctx *ctx, const void *ref, const void *dis,
                     int n_frames, double *scores, void *stream);

/*
 * ss2_score_frames_host — as ss2_score_frames with HOST input pointers.
 * The library uploads the frames itself, batch by batch, on a copy stream
 * into two device slots, so the upload of batch k+1 overlaps the scoring of
 * batch k; an upload into a slot waits on the device for the kernels that
 * last read that slot.  Page-locked (pinned) host memory gives asynchronous
 * copies; pageable memory works but copies synchronously.
 */
int ss2_score_frames_host(ss2_ctx *ctx, const void *ref_host,
                          const void *dis_host, int n_frames, double *scores,
                          void *stream);

/*
 * ss2_values — as ss2_score_frames, and also returns the 108 pooled values
 * of every frame (values: HOST array, n_frames * 108 doubles, index
 * ((c * 6 + s) * 2 + n) * 3 + k for channel c (X, Y, B), scale s, norm n
 * (0: mean, 1: fourth root of the mean fourth power) and map k (0: SSIM,
 * 1: artifact, 2: detail lost); scales that are not computed hold 0).
 * scores may be NULL.
 */
int ss2_values(ss2_ctx *ctx, const void *ref, const void *dis, int n_frames,
               double *values, double *scores, void *stream);

/*
 * ss2_debug_planes — runs the pipeline on one frame pair (device pointers)
 * and copies intermediate planes of one scale to host memory, packed
 * (no pitch).  Any output pointer may be NULL.
 *   xyb:   6 planes ws*hs: ref X, Y, B then dis X, Y, B
 *   hblur: 15 planes: per channel, (mu1, mu2, s11, s22, s12) after the
 *          horizontal recursive pass
 * Returns -EINVAL for a scale the geometry does not reach.
 */
int ss2_debug_planes(ss2_ctx *ctx, const void *ref, const void *dis,
                     int scale, float *xyb, float *hblur, void *stream);

/*
 * ss2_debug_linear — runs the pyramid kernel on one frame pair (device
 * pointers) and copies the linear RGB of one scale to host memory: the
 * YUV -> linear RGB conversion at scale 0 (picture_to_linear_rgb), and the
 * 2x2 downsample of linear RGB at scales 1-5 (downsample_2x2; Research-1363,
 * "Sources" and Finding 2), which the kernel otherwise keeps on chip.
 *   lin: HOST array of 6 planes ws*hs, packed: ref R, G, B then dis R, G, B.
 * The device buffer for the planes is allocated and freed inside the call.
 * Returns -EINVAL for a scale the geometry does not reach or a NULL output.
 */
int ss2_debug_linear(ss2_ctx *ctx, const void *ref, const void *dis, int scale,
                     float *lin, void *stream);

/*
 * ss2_debug_cbrt — applies the pipeline's correctly rounded cube root
 * (linear_rgb_to_xyb's cbrtf; Research-1363, Finding 2) to n floats.
 * x, y: DEVICE arrays of n floats (may alias).  Non-negative finite inputs
 * get cbrt rounded to nearest; other inputs are copied.  Synchronises
 * stream before returning.
 */
int ss2_debug_cbrt(const float *x, float *y, long long n, void *stream);

/*
 * ss2_debug_cbrt_host — the host's correctly rounded cube root, the one that
 * sets the three cbrt(bias_i) constants of the XYB conversion (Research-1363,
 * Finding 2) whenever parameters are set.  x, y: HOST arrays of n floats
 * (may alias); every finite input, of either sign, gets cbrt rounded to
 * nearest (odd: cbrt(-x) = -cbrt(x), zeros keep their sign); infinities and
 * NaN are copied.  Needs no GPU.  Returns -EINVAL for a NULL array with
 * n > 0 or a negative n.
 */
int ss2_debug_cbrt_host(const float *x, float *y, long long n);

/*
 * ss2_set_graphs — how ss2_score_frames and ss2_values launch their work
 * (CUDA graphs, a launch mechanism, not a step of the method).
 * enable = 0 (the default): every kernel is launched one by one.
 * enable != 0: a context's first device-input call launches its kernels
 * one by one; a later call captures the call's whole launch
 * sequence (both lanes' kernels, the score and value read-backs and the
 * error-word read) as a CUDA graph on a stream of the context's own, then
 * replays it with one graph launch on the caller's stream, and so do the
 * calls after it while the frame pointers, the frame count, the outputs
 * asked for and the profiling state stay the same; any change captures
 * again, and ss2_set_params drops the graph.  A capture that the runtime
 * refuses returns the context to one-by-one launches.  The kernels and
 * their inputs are the same in both modes, so are the results, bit for bit.
 * With ss2_profile_begin on, the captured launches carry timing events and
 * ss2_profile_end counts them like the others.  ss2_score_frames_host
 * always launches one by one.  Replays measured no faster on GB300 at the
 * sizes tried, 576x324 to 3840x2160 (a call's time is its kernels' serial
 * walks, not their launches), hence the default.  Returns 0, or -EINVAL for
 * a NULL context.
 */
int ss2_set_graphs(ss2_ctx *ctx, int enable);

/*
 * ss2_profile_begin / ss2_profile_end — per-kernel device timing.  Between
 * the two calls every kernel launch of the context is bracketed by a pair of
 * CUDA events on its launching stream.  ss2_profile_end waits for those
 * events and writes, per kernel class (0 k_pyramid, 1 k_hblur, 2 k_vblur,
 * 3 k_finalize), the summed milliseconds (ms, 4 doubles) and the number of
 * launches (launches, 4 ints); either pointer may be NULL.
 */
int ss2_profile_begin(ss2_ctx *ctx);
int ss2_profile_end(ss2_ctx *ctx, double *ms, int *launches);

/*
 * ss2_debug_wait_probe — runs a one-warp kernel whose shared-memory barrier
 * phase is never completed and lets its bounded wait give up after `spins`
 * polls (the same bounded wait the TMA kernels use).  Returns -EIO when the
 * kernel reported the timeout (the expected outcome), 0 if the wait
 * completed, another negative code on a CUDA error.  Synchronises stream.
 * The device stays usable afterwards.
 */
int ss2_debug_wait_probe(unsigned spins, void *stream);

/* ss2_frame_bytes — bytes of one packed frame of the context's geometry. */
size_t ss2_frame_bytes(const ss2_ctx *ctx);

/* ss2_batch — frames processed per pass (each workspace's batch size).   */
int ss2_batch(const ss2_ctx *ctx);

/* ss2_workspace_bytes — device bytes the context holds.                  */
size_t ss2_workspace_bytes(const ss2_ctx *ctx);

/*
 * Parameter vector (SS2_NPARAMS doubles):
 *   [0, 108)   pooling weights w_i (index as in ss2_values)
 *   [108, 112) polynomial p0..p3: score = p0 + p1 P + p2 P^2 + p3 P^3,
 *              P = sum_i w_i |v_i|
 *   [112, 115) power map alpha, beta, gamma: if score > 0,
 *              score = alpha * score^beta + gamma (beta == 1: no pow)
 *   [115, 124) 3x3 opsin mixing matrix, row-major
 *   [124, 127) opsin biases (must be > 0)
 *   [127, 132) make-positive affine sx, ox, oy, sb, ob:
 *              X' = sx X + ox, Y' = Y + oy, B' = (B - Y) sb + ob
 *   [132]      SSIM stabiliser C2
 * The fp32 pipeline uses each value rounded to float once.  Defaults: the
 * XYB opsin matrix and bias of JPEG XL (ISO/IEC 18181-1) and C2 = 0.0009;
 * placeholders for the tuned SSIMULACRA2 constants, which the source pages
 * do not give (weights 1/108, score = 100 - 100 P, identity affine).
 */
int ss2_default_params(double *params, int n_params);
int ss2_set_params(ss2_ctx *ctx, const double *params, int n_params);

/* ss2_host_tables — the library's own host-built constant tables, for
 * checks without a device: eotf (4097 floats, the sRGB EOTF on a uniform
 * grid of 4096 intervals) and iir (6 floats: 2 cos(w_k) for k = 1, 3, 5,
 * then a_k cos(4 w_k), the recursive Gaussian's coefficients).  Either
 * pointer may be NULL.                                                     */
int ss2_host_tables(float *eotf, float *iir);

/*
 * ss2_score_frames_noalloc — scores n_frames frame pairs without allocating
 * anything, for callers that cannot call cudaMalloc at scoring time (code
 * inside a custom allocator or memory-pool callback, processes with a device
 * memory budget fixed up front, plug-ins handed buffers by a host that
 * forbids allocation).  It has no counterpart on the source pages: it is the
 * ss2_score_frames path with its workspace in one fixed 64 MiB device array
 * that the library holds on every GPU that loads it, until exit.
 *   width, height, bitdepth, chroma: as ss2_create; the frame's workspace
 *             must fit the 64 MiB array (about 600k pixels, e.g. 853x481 or
 *             960x540), else -EINVAL before any GPU work.
 *   ref, dis: DEVICE pointers to n_frames packed frames each (caller-owned).
 *   scores:   DEVICE array of n_frames doubles (caller-owned), written by the
 *             last kernel; the call does not synchronise or read back.
 *   stream:   cudaStream_t for all work (NULL = legacy default stream).
 * Uses the default parameters.  The first call on a device does a one-time
 * set-up (looks up the array's address, copies the constant tables with
 * synchronous copies); make it before any stream capture.  All calls on a
 * device share the array and keep the last call's contents; calls that
 * overlap on the GPU race and corrupt each other's results.  Each call
 * first clears the array's error word on `stream` (a memset, which
 * allocates nothing).  A kernel whose bounded wait for a copy runs out sets
 * that word; the call cannot see it (it reads nothing back), so the scores
 * of the batch then being scored, and of every later batch of the call, are
 * written as NaN: check the scores for NaN where that matters.  The set-up
 * is kept for the life of the process: do not use this entry point after a
 * cudaDeviceReset of a device it ran on.  Returns 0 or a negative code as
 * the other entry points.
 */
int ss2_score_frames_noalloc(int width, int height, int bitdepth, int chroma,
                             const void *ref, const void *dis, int n_frames,
                             double *scores, void *stream);

/* ss2_debug_noalloc_timeout — test hook of ss2_score_frames_noalloc (no
 * counterpart on the source pages): with spins > 0, every later call first
 * runs a one-warp bounded wait on a barrier phase that nothing completes
 * (spins polls), which gives up and sets the call's error word, so that the
 * NaN signal above can be checked without faulting anything; 0 turns it off.
 * Returns 0.                                                               */
int ss2_debug_noalloc_timeout(unsigned spins);

/*
 * float_ssim with decimation on the device ("ADR-1405: float_ssim_hip
 * decimates on the device, bit-identical to the CPU", Context and Decision
 * 1 and 4).  The luma plane of each frame (the same packed frames as above;
 * chroma is not read), in the 8-bit range (raw / 2^(depth - 8)), is
 * decimated by max(1, round(min(w, h) / 256)): a scale x scale box of weight
 * RN(1 / scale^2) at (x * scale, y * scale), offsets -scale/2 ..
 * scale-1-scale/2, symmetric edges, the fp32 taps summed exactly (int64
 * units of 2^-52) and rounded once; then SSIM with an 11x11 Gaussian window
 * (sigma 1.5, K1 = 0.01, K2 = 0.03, L = 255) over the positions where the
 * window fits, averaged.
 *   ss2_fssim_create: geometry as ss2_create; max_batch 0 = 64 frames per
 *     pass.  NULL with -ENOTSUP when the decimated plane is below 11x11 or
 *     the factor exceeds 128, -EINVAL for bad geometry.
 *   ss2_fssim_score: ref, dis DEVICE frames (n_frames packed frames each,
 *     owned by the caller, read only); scores HOST doubles (n_frames); one
 *     stream synchronisation per call.  0 on success; -EINVAL for a NULL
 *     context or pointer or a negative count (0 frames: no work); -ENOMEM
 *     when the pinned staging cannot grow; -EIO on a CUDA failure.  The
 *     context owns its workspace: 2 fp32 planes of pitch x ceil(h/scale)
 *     (pitch = ceil(w/scale) rounded up to 32) per frame of the batch.
 *   ss2_fssim_scale: the decimation factor.
 *   ss2_fssim_debug_decimated: the two decimated planes of one frame pair
 *     (HOST floats, ref then dis, each ceil(w/scale) x ceil(h/scale),
 *     packed).
 *   ss2_fssim_profile_begin / _end: as ss2_profile_begin / _end, kernel
 *     classes 0 k_fssim_decimate, 1 k_fssim_map, 2 k_fssim_final (ms: 3
 *     doubles, launches: 3 ints, either may be NULL).
 */
typedef struct ss2_fssim ss2_fssim;
ss2_fssim *ss2_fssim_create(int width, int height, int bitdepth, int chroma,
                            int max_batch);
int ss2_fssim_score(ss2_fssim *ctx, const void *ref, const void *dis,
                    int n_frames, double *scores, void *stream);
int ss2_fssim_scale(const ss2_fssim *ctx);
int ss2_fssim_debug_decimated(ss2_fssim *ctx, const void *ref,
                              const void *dis, float *planes, void *stream);
int ss2_fssim_profile_begin(ss2_fssim *ctx);
int ss2_fssim_profile_end(ss2_fssim *ctx, double *ms, int *launches);
void ss2_fssim_destroy(ss2_fssim *ctx);

/*
 * MS-SSIM of the luma plane ("Research-1363: Device-resident ssimulacra2 and
 * a single-wait MS-SSIM on SYCL", Findings 6 and 9; the method of Wang,
 * Simoncelli and Bovik, "Multi-scale structural similarity for image quality
 * assessment", 2003).  Samples in the 8-bit range (raw / 2^(depth - 8));
 * five scales, scale j + 1 the 2x2 mean of scale j with the edge sample
 * repeated (ceil halving); at every scale the 11x11 Gaussian (sigma 1.5)
 * SSIM statistics wherever the window fits, K1 = 0.01, K2 = 0.03,
 * C3 = C2 / 2, L = 255, and the means of l, c, s, cs and l cs; the score
 * prod_{j<5} mean(cs_j)^beta_j * mean(l cs)_5^beta_5, beta = (0.0448,
 * 0.2856, 0.3001, 0.2363, 0.1333).  All scales of a batch are enqueued at
 * once; one stream synchronisation per call.
 *   ss2_msssim_create: geometry as ss2_create; max_batch 0 = 32 frames per
 *     pass; the luma plane only.  NULL with -ENOTSUP when the scale-5 plane
 *     is below 11x11 (a side below 161), -EINVAL for bad geometry, -ENOMEM.
 *   ss2_msssim_create_ex: as ss2_msssim_create; enable_chroma != 0 also
 *     scores the Cb and Cr planes (Finding 6 lists enable_chroma among the
 *     outputs), each on its own at chroma resolution (ceil(w / 2^sx) x
 *     ceil(h / 2^sy)) with the same method: NULL with -ENOTSUP when a
 *     chroma plane's scale-5 plane is below 11x11.
 *   ss2_msssim_planes: the planes a context scores, 1 or 3 (-EINVAL for
 *     NULL).
 *   ss2_msssim_score: ref, dis DEVICE frames (n_frames packed frames each,
 *     owned by the caller, read only); scores HOST doubles (n_frames x
 *     planes, frame-major: Y then Cb, Cr); values HOST doubles (n_frames x
 *     planes x 5 scales x (l, c, s, cs, l cs)) or NULL.  0 on success;
 *     -EINVAL for a NULL context or pointer or a negative count (0 frames:
 *     no work); -ENOMEM when the pinned staging cannot grow; -EIO on a CUDA
 *     failure.  The context owns its workspace: per plane, scales 2..5 of
 *     both images (fp32, rows padded to 32 floats) and the per-(frame,
 *     scale, tile) partial sums of each frame of the batch.
 *   ss2_msssim_debug_pyramid: scales 2..5 of the luma plane of one frame
 *     pair (HOST floats: ref scales 2..5 then dis scales 2..5, each w_j x
 *     h_j packed); ss2_msssim_debug_pyramid_plane: the same for plane 0, 1
 *     or 2 (-EINVAL for a plane the context does not score).
 *   ss2_msssim_profile_begin / _end: as ss2_profile_begin / _end, kernel
 *     classes 0 k_msssim_level (all scales), 1 k_msssim_final (ms: 2
 *     doubles, launches: 2 ints, either may be NULL).
 */
typedef struct ss2_msssim ss2_msssim;
ss2_msssim *ss2_msssim_create(int width, int height, int bitdepth, int chroma,
                              int max_batch);
ss2_msssim *ss2_msssim_create_ex(int width, int height, int bitdepth, int chroma,
                                 int max_batch, int enable_chroma);
int ss2_msssim_planes(const ss2_msssim *ctx);
int ss2_msssim_score(ss2_msssim *ctx, const void *ref, const void *dis,
                     int n_frames, double *scores, double *values, void *stream);
int ss2_msssim_debug_pyramid(ss2_msssim *ctx, const void *ref, const void *dis,
                             float *planes, void *stream);
int ss2_msssim_debug_pyramid_plane(ss2_msssim *ctx, const void *ref, const void *dis,
                                   int plane, float *planes, void *stream);
int ss2_msssim_profile_begin(ss2_msssim *ctx);
int ss2_msssim_profile_end(ss2_msssim *ctx, double *ms, int *launches);
void ss2_msssim_destroy(ss2_msssim *ctx);

/*
 * CAMBI c-values and top-K pooling ("ADR-1357: Run the SYCL CAMBI extractor
 * entirely on the device", Decision).  The stages before them (10-bit
 * conversion, spatial mask, decimation, mode filter) are the caller's: a
 * plane here is a w x h array of 10-bit levels (uint16, < 1024, rows packed)
 * with an optional mask (uint8, nonzero = counted, same layout).
 *   c-value of a counted pixel of level L: the largest over the (d, w) table
 *     of (float)(w p0 pm) * RN(1 / (p0 + pm)), with p0 and pm the counts of
 *     levels L and L + d among the counted pixels of the window x window
 *     square centred on it, clipped to the plane (a term with pm = 0 is 0);
 *     0 for a pixel that is not counted.  Every nonzero value lies in
 *     [0.5, 2^14) and so on the 2^-24 grid.
 *   top-K pool of a plane's c-values: T the k-th largest, the exact sum
 *     S = sum(v > T) + (k - #(v > T)) T in units of 2^-24 (128 bits), the
 *     mean S 2^-24 / k in fp64.
 *   ss2_cambi_create: window odd with window^2 <= 4225 (at most 65), 1..4
 *     (diff, weight) pairs (diff 1..1023, weight 1..9), max_batch 0 = as
 *     many planes per pass as 2 GB of c-values hold, 1 to 64 (at most 1024
 *     when given).  NULL with -EINVAL for bad arguments, -ENOMEM.
 *   ss2_cambi_cvalues: levels (and mask, or NULL) DEVICE, n_planes planes;
 *     cvalues DEVICE floats, n_planes planes.  -EINVAL for a level >= 1024.
 *   ss2_cambi_topk: cvalues DEVICE (values 0 or on the 2^-24 grid below
 *     2^14, else -EINVAL); k in 1..w h; sums HOST (lo, hi) pairs of
 *     uint64, thresholds HOST floats, means HOST doubles, n_planes each;
 *     any output pointer may be NULL.
 *   ss2_cambi_pool: both stages, the c-values kept in the context's own
 *     workspace; outputs as ss2_cambi_topk.
 *   All three: 0 on success, -EINVAL (NULL context or input, negative
 *   count; 0 planes: no work), -ENOMEM (pinned staging), -EIO (CUDA
 *   failure); one stream synchronisation per call.  The context owns its
 *   workspace (one batch of c-values, radix histograms, block sums).
 *   ss2_cambi_profile_begin / _end: kernel classes 0 k_cambi_cvalues, 1 the
 *     top-K kernels (ms: 2 doubles, launches: 2 ints, either may be NULL).
 */
typedef struct ss2_cambi ss2_cambi;
ss2_cambi *ss2_cambi_create(int width, int height, int window, int ndiff,
                            const int *diffs, const int *weights, int max_batch);
int ss2_cambi_cvalues(ss2_cambi *ctx, const uint16_t *levels, const uint8_t *mask,
                      int n_planes, float *cvalues, void *stream);
int ss2_cambi_topk(ss2_cambi *ctx, const float *cvalues, int n_planes, long long k,
                   uint64_t *sums, float *thresholds, double *means, void *stream);
int ss2_cambi_pool(ss2_cambi *ctx, const uint16_t *levels, const uint8_t *mask,
                   int n_planes, long long k, uint64_t *sums, float *thresholds,
                   double *means, void *stream);
int ss2_cambi_profile_begin(ss2_cambi *ctx);
int ss2_cambi_profile_end(ss2_cambi *ctx, double *ms, int *launches);
void ss2_cambi_destroy(ss2_cambi *ctx);

/* Last failure on the calling thread (0 if none yet).                      */
int ss2_last_error(void);
const char *ss2_last_error_string(void);

#ifdef __cplusplus
}
#endif
#endif
