/*
 * sscan_tuning.h -- layout overrides and a fault-injection hook for libsscan. For tests and
 * tuning sweeps; normal callers never need it (the pages define no such controls; they exist so
 * that tests can force every kernel layout and the chunk-carry timeout path).
 *
 * The library chooses its kernel layout from the problem shape. sscan_set_tuning replaces those
 * choices, process-wide, for every later call on any device until it is called again; a field
 * left at 0 (-1 for test_skip_publish) keeps the automatic choice. Nothing else (no environment
 * variable, no file) changes what the library does. Calls already launched are not affected.
 * Thread safety: the setting is read once per call under a lock; changing it while other host
 * threads are calling the library is allowed but makes which setting those calls see undefined.
 */
#ifndef SSCAN_TUNING_H
#define SSCAN_TUNING_H

#include "sscan.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int states_per_lane;   /* forward: states of one channel a lane holds: 16, 8 or 4 (0: auto) */
  int segments;          /* forward: time segments of one sequence run by different thread
                            blocks, joined by the chunk carry (0: auto; 1: never split) */
  int threads;           /* forward: threads per block, a multiple of 32 up to 256 (0: auto) */
  int stages;            /* forward: TMA pipeline depth, 2..8 (0: auto) */
  int chunk;             /* forward, four lanes per channel: steps per chunk, 16 or 32 (0: auto) */
  int force_plain;       /* forward: 1 = always the plain-load kernel (0: TMA path when possible) */
  int bwd_segments;      /* backward: time segments (0: auto) */
  int conv_plain;        /* Conv1d: 1 = always the register-window kernel (0: TMA when possible) */
  int ctas_per_sm;       /* forward: at most this many thread blocks resident per SM, 1..32
                            (enforced through each block's shared-memory reservation; 0: auto) */
  int test_skip_publish; /* fault injection: the time segment with this index never publishes
                            its chunk-carry summary, so that its successors' bounded waits run
                            out and report SSCAN_ERR_CARRY_TIMEOUT (-1: off) */
  int time_scan;         /* forward: 1 = the time-lane kernel (a warp scans one channel over
                            time, the lanes' aggregates composed in order), 2 = never, 0 = auto
                            (at most 64 channels, or at most 256 channels and 2^23 channel-steps,
                            unless states_per_lane, threads or chunk is set); calls that write
                            backward checkpoints never use it */
} sscan_tuning_t;

/* Installs *t (NULL: back to every automatic choice, hook off). Returns SSCAN_ERR_INVALID_ARG
 * for a field outside the ranges above (the setting is then unchanged), else SSCAN_OK. */
sscan_status_t sscan_set_tuning(const sscan_tuning_t* t);

/* Copies the current setting into *t (SSCAN_ERR_INVALID_ARG if t is NULL). */
sscan_status_t sscan_get_tuning(sscan_tuning_t* t);

/* y[i] = 2^x[i] for i < n (device memory, fp32, asynchronous on `stream`), computed with the
 * library's own accurate exponential: the one the fp32 path uses to re-anchor the decay over a
 * chunk, exp(dt A) over the chunk's summed step (zero-order hold of "架构变体：Mamba/SSM",
 * section "离散化"). Arguments are clamped to [-125, 125]. Exposed so that tests can check its
 * accuracy and its lack of bias against the exact exponential. n = 0 is a no-op; x or y NULL
 * with n > 0, or n < 0, returns SSCAN_ERR_INVALID_ARG. */
sscan_status_t sscan_exp2_accurate(const float* x, float* y, int64_t n, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SSCAN_TUNING_H */
