// Minimal arbitrary-precision naturals for the host reconstruction stage
// (64-bit limbs, little-endian, no leading zero limbs; zero = empty).
// Schoolbook and Karatsuba multiplication, Knuth's Algorithm D division,
// Lehmer's extended Euclid (optionally on helper threads), half-gcd stages.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

namespace es {
namespace big {

using limb = uint64_t;
using Nat = std::vector<limb>;

void trim(Nat& a);
int cmp(const Nat& a, const Nat& b);
size_t bitlen(const Nat& a);
bool is_zero(const Nat& a);
Nat from_u64(uint64_t v);
Nat add(const Nat& a, const Nat& b);
Nat sub(const Nat& a, const Nat& b);  // a >= b
void add_in(Nat& a, const Nat& b);
void sub_in(Nat& a, const Nat& b);  // a >= b
Nat mul(const Nat& a, const Nat& b);
Nat mul_small(const Nat& a, limb s);
void mul_small_add_in(Nat& a, const limb* s, int slen, const limb* add, int alen);  // a = a*s + add
void divmod(const Nat& u, const Nat& v, Nat* q, Nat* r);                            // v != 0
Nat shl(const Nat& a, size_t bits);
Nat shr(const Nat& a, size_t bits);
// a <= 2^k
bool le_pow2(const Nat& a, size_t k);

// A cofactor pipe lets a second thread follow the cofactors of one
// rational_reconstruct run (ReconOpts::pipe): that thread calls
// cofactor_pipe_serve() beside the run -- before, during or after it -- and
// returns once the run is over.  Whichever side claims the work first does
// it, so the run never waits for a server that has not started.  One pipe
// per run; a pipe is used once.
struct CofactorPipe;
CofactorPipe* cofactor_pipe_new();  // null when out of memory
void cofactor_pipe_free(CofactorPipe* p);
void cofactor_pipe_serve(CofactorPipe* p);
// Ends serve() calls once nothing is left for them (a run closes its pipes
// itself on every way out; closing again is harmless).
void cofactor_pipe_close(CofactorPipe* p);
// A low-limb pipe lets a further thread take the low limbs of the remainders
// of one run that has a cofactor pipe (ReconOpts::low): the run updates the
// high limbs from each batch's matrix and that thread follows over the low
// ones, a bounded number of batches behind.  The run splits the work only
// while a thread serves the pipe (low_pipe_serve, before, during or after the
// run; it returns once the run is over).  One pipe per run, used once.
struct LowPipe;
LowPipe* low_pipe_new();  // null when out of memory
void low_pipe_free(LowPipe* p);
void low_pipe_serve(LowPipe* p);
void low_pipe_close(LowPipe* p);  // as cofactor_pipe_close
// How rational_reconstruct runs.  pipe: its Lehmer loop hands the cofactor
// updates to whoever serves the pipe; low (with pipe only): the low limbs of
// the remainders likewise.  hgcd_min_bits: from this length of M on,
// half-gcd stages (subquadratic) do most of the reduction.  They are off by
// default: alone they beat the Lehmer loop only from about 10^5 bits (167 K
// bits: 7.8 against 9.6 ms on the Grace host), and their many short-lived
// products scale badly when a whole pool of reconstructions runs at once
// (sixteen at 166 K bits took 52-75 ms each).
struct ReconOpts {
  CofactorPipe* pipe = nullptr;
  LowPipe* low = nullptr;
  size_t hgcd_min_bits = SIZE_MAX;
};
// Extended Euclid on (r0 = M, r1 = u) stopped at the first remainder <= 2^nbits
// (Wang's rational reconstruction).  Returns den = |t| and num = r with its
// sign (num_neg), or false when no remainder ever gets that small.  The
// result does not depend on opts.
bool rational_reconstruct(const Nat& M, const Nat& u, size_t nbits, Nat* num, bool* num_neg, Nat* den,
                          const ReconOpts& opts = ReconOpts());
Nat gcd(const Nat& a, const Nat& b);

}  // namespace big
}  // namespace es
