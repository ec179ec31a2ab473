/*
 * es.h -- C ABI of the GB300 exact rational solver (Dixon p-adic lifting).
 *
 * Solves integer systems A x = b exactly over the rationals, as defined by
 * the exact-solve card (kernels hub), §API: the solution of A [n, n] x = b
 * [n, c] returned as numerators and a denominator, or "singular" when A is
 * singular over Q.  The method is the card's §Method: Dixon lifting over the
 * squarefree modulus P = prod q_j of the odd primes q_j < 256, with
 *   B_j = A^{-1} mod q_j by batched Gauss-Jordan (Barrett reduction),
 *   x_i = B r_i mod P per prime + balanced Garner/CRT into one wide digit,
 *   r_{i+1} = (r_i - A x_i) P^{-1} mod 2^64 in one signed 64-bit limb,
 * stopping once P^m > 2 N_H D_H (Hadamard bounds on numerator and
 * denominator), then rational reconstruction from x mod P^m.
 *
 * Conventions shared by every entry point
 *   - Matrices are row-major.  Host pointers are read during the call only
 *     and never retained.  Device pointers must be device-accessible memory
 *     of the current CUDA device.
 *   - Range (card, §Method "Range" and §Requirements): n >= 1, c >= 1,
 *     n <= 2^17 and n * max|A_ij| < 2^63 (strict); otherwise ES_ERR_RANGE.
 *   - Nothing aborts or throws across this boundary: every failure is a
 *     status code.  CUDA errors are reported as ES_ERR_CUDA with the CUDA
 *     error text available from es_last_error().
 *   - Calls are synchronous with respect to the host (they return after the
 *     device work they issued has finished).  Device work is ordered on the
 *     caller's stream (es_options.stream, or a library stream when NULL).
 *   - The library keeps one device workspace per device, grown on demand
 *     and reused across calls (es_release_workspace() frees it).  Calls on
 *     the same device must not overlap in time (one solve at a time per
 *     device); the library serialises them with a mutex.
 *   - Primes are indexed 0..52 in ascending order (3, 5, 7, ..., 251).
 */
#ifndef EXACT_SOLVE_ES_H
#define EXACT_SOLVE_ES_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ES_NUM_PRIMES 53 /* odd primes below 256 */
#define ES_DIGIT_LIMBS 6 /* one balanced base-P digit: 6 x 64-bit two's complement */
#define ES_NUM_PHASES 6  /* see es_solution_phase_ms */

typedef enum {
  ES_OK = 0,
  ES_SINGULAR = 1,      /* A singular over Q (card §API: solve returns None) */
  ES_ERR_ARG = -1,      /* null pointer, bad size or option */
  ES_ERR_RANGE = -2,    /* outside n <= 2^17, n * max|A_ij| < 2^63 */
  ES_ERR_CUDA = -3,     /* a CUDA runtime call failed (es_last_error has the text) */
  ES_ERR_NOMEM = -4,    /* device or host allocation failed, or max_device_bytes exceeded */
  ES_ERR_TIMEOUT = -5,  /* a kernel's bounded wait ran out (its error flag was set), or fault injection */
  ES_ERR_INTERNAL = -6, /* a self-check failed (e.g. a reconstruction bound) */
  ES_ERR_NODEVICE = -7  /* no CUDA device visible */
} es_status;

typedef struct es_options {
  void* stream;            /* cudaStream_t to order device work on; NULL = library stream */
  size_t max_device_bytes; /* 0 = no cap; else ES_ERR_NOMEM when the workspace would exceed it */
  int32_t fault_stage;     /* fault injection: 0 = none, else see ES_FAULT_* */
  int32_t threads;         /* host threads for reconstruction; 0 = all hardware threads */
  int32_t timing;          /* 1: time each phase with CUDA events; 2: also time every launch
                              of the lift's per-prime product kernel (es_solution_kernels) */
  int32_t flags;           /* bit set of ES_FLAG_* */
} es_options;

/* es_options.flags */
#define ES_FLAG_HOST_RECON 1 /* reconstruct on the host even when the GPU numerator pass applies */
#define ES_FLAG_STEP_LIFT 2  /* c == 1: run the lift as per-step kernels instead of the fused launch */
#define ES_FLAG_ONE_STREAM 4 /* run the inverse on the caller's stream alone, without the two SM partitions */

/* Fault injection points (es_options.fault_stage): the named stage returns
 * the given status without running; used to test error propagation. */
#define ES_FAULT_RESIDUES 1  /* -> ES_ERR_CUDA */
#define ES_FAULT_INVERSE 2   /* -> ES_ERR_CUDA */
#define ES_FAULT_LIFT 3      /* -> ES_ERR_TIMEOUT */
#define ES_FAULT_RECON 4     /* -> ES_ERR_INTERNAL */
#define ES_FAULT_NOMEM 5     /* -> ES_ERR_NOMEM at workspace allocation */
#define ES_FAULT_LIFT_WAIT 6 /* device side: the fused lift (c == 1, n <= 1024) starts its grid-barrier
                                counter where the first barrier can never complete; every CTA's
                                bounded wait (2 s) expires, the kernel returns -> ES_ERR_TIMEOUT */

typedef struct es_solution es_solution; /* opaque, owned by the library */

/* ---------------------------------------------------------------- solve
 * es_solve: exact solution of A x = b (card §API, solve(A, b)).
 *   A    host int64 [n, n], row-major;  b  host int64 [n, c], row-major.
 *   opt  may be NULL (defaults).
 *   out  receives a solution handle on ES_OK; set to NULL otherwise
 *        (ES_SINGULAR included).  Free with es_solution_free().
 * The result is canonical: one common denominator d > 0 for all n*c
 * entries, the least with d*x integral, and numerators N = d*x.
 * Host->device copies of A and b and the device->host copy of the digits
 * are part of the call.
 */
es_status es_solve(const int64_t* A, const int64_t* b, int64_t n, int64_t c,
                   const es_options* opt, es_solution** out);

/* es_solve_device: as es_solve with A and b already in device memory
 * (e.g. torch tensors on the current CUDA device), read on opt->stream. */
es_status es_solve_device(const int64_t* A_dev, const int64_t* b_dev, int64_t n, int64_t c,
                          const es_options* opt, es_solution** out);

/* Shape of a solution: n, c, and the number of 64-bit limbs of every
 * exported numerator and of the denominator (wide enough for both). */
es_status es_solution_shape(const es_solution* s, int64_t* n, int64_t* c, int64_t* limbs);

/* Export: num [n*c*limbs] (entry (i, j) at ((i*c + j) * limbs), little-endian
 * two's complement limbs), den [limbs] (little-endian, > 0).  Host buffers
 * owned by the caller. */
es_status es_solution_export(const es_solution* s, uint64_t* num, uint64_t* den);
/* The same limbs in place: *num ([n*c][limbs]) and *den ([limbs]) point into
 * the solution and stay valid until es_solution_free (no copy).  Any
 * pointer may be NULL; ES_ERR_ARG for a NULL solution. */
es_status es_solution_data(const es_solution* s, const uint64_t** num, const uint64_t** den);

/* Phase times in ms (ms[ES_NUM_PHASES], any may be NULL):
 *   0 range check + bounds + residues, 1 modular inverse, 2 lift,
 *   3 digits device->host (host reconstruction only), 4 rational
 *   reconstruction (sampled denominators on the host + numerator pass on the
 *   GPU, or all on the host), 5 total.
 * Phases 0-3 are filled only when es_options.timing was set; 4 and 5
 * always.  m = lift steps, primes_used = primes not dividing det A. */
es_status es_solution_phase_ms(const es_solution* s, double* ms, int32_t* m, int32_t* primes_used);

/* Kernel accounting of the solve: launches = device kernels the library
 * launched for it; for the dominant kernel of the lift (named by
 * es_solution_top_kernel): its launch count, the summed CUDA-event duration
 * of those launches in ms (only with es_options.timing == 2, else 0), and
 * its algorithmic bytes per launch:
 *   k_lift_fused (c == 1, n <= 1024: all m steps in one launch):
 *     m (E' n^2 + w_A n^2 + n (8 + E' + 48)), w_A = 4 or 8 bytes per entry of A
 *   per-step product kernels (B_j R_j of every good prime):
 *     E' (n^2 + 2 n c)
 * Any pointer may be NULL. */
es_status es_solution_kernels(const es_solution* s, int64_t* launches, int64_t* top_launches, double* top_ms,
                              double* top_bytes_per_launch);

/* Name of that dominant lift kernel ("k_lift_fused", "k_lift_gemv",
 * "k_lift_gemm" or "k_lift_gemm_tc"); a static string, "" for NULL. */
const char* es_solution_top_kernel(const es_solution* s);
/* 1 when the solve's modular inverse ran on two SM partitions (green
 * contexts: the next column block's panels on 56 SMs while the previous
 * block's update uses the rest), 0 when it ran on the solve's stream alone
 * (ES_FLAG_ONE_STREAM, n > 1024, or no green-context support); 0 for NULL. */
int32_t es_solution_inverse_split(const es_solution* s);

void es_solution_free(es_solution* s);

const char* es_status_string(es_status st);
/* Text of the last CUDA error seen by this thread ("" if none). */
const char* es_last_error(void);
/* Frees the device workspace and cached graphs of the current device. */
es_status es_release_workspace(void);
/* Library ABI version (bumped on incompatible changes). */
int32_t es_version(void);

/* ---------------------------------------------------------------- stages
 * Stage-level entry points on device buffers, ordered on `stream` (a
 * cudaStream_t, NULL = library stream) and synchronous on return.  They are
 * the stages es_solve runs, exposed for checking and for callers that keep
 * the inverse across right-hand sides.
 */

/* Balanced residues (card §Method: per-prime products run on balanced
 * residues): out[j][i] = A[i] mod q_j in [-(q_j-1)/2, (q_j-1)/2] for
 * i < count, j < 53.  A_dev int64 [count]; out_dev int8 [53][count]. */
es_status es_residues_device(const int64_t* A_dev, int64_t count, int8_t* out_dev, void* stream);

/* Batched modular inverse (card §Method: A^{-1} mod q_j for every prime by
 * Gauss-Jordan, one grid per elimination step spanning all primes, Barrett
 * reduction).  A_dev int64 [n, n].  Writes B_dev int8 [53][n][ld] with
 * ld = (n + 15) / 16 * 16: B_dev[j][i][k] = (A^{-1} mod q_j)[i][k], balanced,
 * zero in the padding columns k >= n; and good_dev uint8 [53]: 1 when q_j
 * does not divide det A (B_j valid), 0 otherwise (B_j unspecified).
 * Range rules apply to A (ES_ERR_RANGE). */
es_status es_inverse_mod_device(const int64_t* A_dev, int64_t n, int8_t* B_dev, uint8_t* good_dev,
                                void* stream);

/* Batched modular inverse that allocates nothing (the card has no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory -- code inside a framework whose caching allocator already
 * holds nearly all of it, or latency-bound loops that must not pay the
 * device-wide synchronisation of cudaFree).  Same arguments, layout and
 * result as es_inverse_mod_device for n <= 256; its working memory is a
 * fixed 4.5 MiB array in device memory that every GPU loading the library
 * holds until the process exits.  It calls no cudaMalloc, cudaFree or other
 * allocating routine and creates no stream (NULL = the legacy default
 * stream).  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and should come before
 * any stream capture.  All calls share the array, which keeps the previous
 * call's contents (everything that must start at zero is cleared); calls
 * are serialised on the host, and each returns only after its device work
 * has finished (it synchronises the stream it was given), so device work
 * that overlapped a call on another stream through this array would race.
 * The array's address is looked up once per device and kept for the life of
 * the process: a caller that resets a device (cudaDeviceReset) must not
 * call this entry point on that device again in the same process.
 * Unlike es_inverse_mod_device it accepts any int64 entries (residues are
 * exact for all of them).  n > 256 -> ES_ERR_RANGE with the reason in
 * es_last_error(). */
es_status es_inverse_mod_device_noalloc(const int64_t* A_dev, int64_t n, int8_t* B_dev, uint8_t* good_dev,
                                        void* stream);

/* Lift plan (card §Method stop rule): bit bounds and step count that the
 * solve uses.  num_bits / den_bits: Nb = 2^num_bits >= N_H and
 * Db = 2^den_bits >= D_H with D_H = prod_i ||a_i||_2 and
 * N_H = prod_i sqrt(||a_i||^2 + max_k b_ik^2); m = the least number of steps
 * with P'^m > 2 Nb Db, P' = product of the primes with good[j] != 0.
 * A_dev int64 [n, n], b_dev int64 [n, c], good host uint8 [53]. */
es_status es_plan_device(const int64_t* A_dev, const int64_t* b_dev, int64_t n, int64_t c,
                         const uint8_t* good, int64_t* num_bits, int64_t* den_bits, int32_t* m,
                         void* stream);

/* The lift (card §Method): m Dixon steps from r_0 = b.  Step i writes the
 * balanced base-P' digit x_i (P' = product of primes with good[j] != 0,
 * host uint8 [53]) of every entry to digits_dev uint64 [m][n*c][6]
 * (entry (r, col) at index r*c + col; 6 little-endian two's complement
 * limbs).  B_dev as written by es_inverse_mod_device.  At least one good
 * prime is required (ES_ERR_ARG otherwise). */
es_status es_lift_device(const int64_t* A_dev, const int64_t* b_dev, int64_t n, int64_t c,
                         const int8_t* B_dev, const uint8_t* good, int32_t m, uint64_t* digits_dev,
                         void* stream);

/* Rational reconstruction on the host (card §Method, final stage): from the
 * digits (host uint64 [m][n*c][6], as es_lift_device writes them), the good
 * prime flags and the bit bounds of es_plan_device, the canonical solution:
 * common denominator from a sample of components, then one modular multiply
 * per numerator with an exact acceptance test.  opt may be NULL (threads). */
es_status es_reconstruct(const uint64_t* digits, int64_t n, int64_t c, int32_t m, const uint8_t* good,
                         int64_t num_bits, int64_t den_bits, const es_options* opt, es_solution** out);

/* Host self-check of the library's modular reduction helpers (no GPU):
 * compares the Barrett reduction used by the kernels with the % operator
 * for every odd prime < 256 over all inputs in [lo, hi) of the signed
 * 32-bit accumulator domain, and over `samples` pseudo-random int64
 * values for the 64-bit residue path.  Returns the number of mismatches
 * (0 = pass), or -1 on bad arguments. */
int64_t es_selftest_modular(int64_t lo, int64_t hi, int64_t samples);

/* Host self-check of the reconstruction's big-integer arithmetic (no GPU):
 * `rounds` pseudo-random cases from `seed` (sizes 1..1200 limbs, dense,
 * all-ones and sparse patterns) checking Karatsuba products against a plain
 * schoolbook product, division (q v + r == u, r < v), shifts, and the
 * rational reconstruction's output (num == +-den u mod M, |num| <= 2^nbits,
 * den > 0), and its exact recovery of planted fractions num / den with
 * 2^(nbits+1) den < M (sign included; planted denominators up to 400 limbs).
 * The planted cases, and residues with no small fraction behind them, are
 * reconstructed every way the library can (plain Lehmer loop; cofactors
 * handed to a thread that serves the run's pipe, started before the run or
 * after it; also the remainders' low limbs handed to two more threads;
 * half-gcd stages; combinations), which must agree exactly.  Returns
 * the number of failed checks (0 = pass), or -1 on bad arguments. */
int64_t es_selftest_bigint(uint64_t seed, int64_t rounds);

/* Host self-check of the Gauss-Jordan kernels' f32 residue arithmetic (no
 * GPU; card §Method: the inverse's modular reduction).  The kernels keep row
 * entries as exact f32 integers below 2^20 in magnitude (2^21 + 128 in the
 * depth-128 update) and reduce them as x - q rint(x fl(1/q)) (one fused
 * multiply-add against 1.5 * 2^23, one add, one fused multiply-add); the
 * same source function is run here for every odd prime q < 256 and every
 * integer |x| <= 2^21 + 2^10 and compared with the balanced residue by the %
 * operator, together with the byte extraction that stores the result.
 * Returns the number of mismatches (0 = pass). */
int64_t es_selftest_gj_reduction(void);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_SOLVE_ES_H */
