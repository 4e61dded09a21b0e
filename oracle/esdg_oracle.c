/*
 * CPU ORACLE for the flux-differencing volume term and the surface term of the entropy-stable DG
 * Euler-with-gravity solver in "GPU Performance of an Entropy-Stable
 * Discontinuous Galerkin Euler Solver with Non-Conservative Terms"
 * (Sec. 3 Eq. 2; Sec. 4.1 Eqs. 3-5).
 *
 * TEST INFRASTRUCTURE.  Plain, slow and written to be checked against the
 * paper by eye: full ordered pair sums, no symmetry, no precompute reuse, no
 * blocking.  Only the test suite, the package smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header or table with the
 * CUDA library and includes nothing from it.
 *
 * Two instantiations of the same source: double (suffix _d, the oracle) and
 * long double (suffix _ld, used to measure the double oracle's own rounding).
 *
 * Parity pins (tests/test_oracle_pins.py): consistency with the physical flux
 * of Eq. 1, symmetry and the gravity partner scaling of Sec. 4.1, the pair
 * entropy-conservation condition, per-element conservation and SBP entropy
 * identity, free-stream preservation on curved meshes, a hydrostatic closed
 * form, metric identities and closed forms, and LGL operator identities.
 *
 * The surface term (Eq. 2's M^-1 M^s G^s F*, with F* the entropy-conserving
 * flux plus matrix dissipation) is pinned in tests/test_oracle_surface_pins.py:
 * the eigen-structure and entropy Jacobian against complex-step derivatives
 * of the physical flux and entropy variables, the Roe small-jump limit,
 * entropy stability, conservation, free stream, and the global entropy
 * balance of volume + surface.
 */
#include <stdlib.h>
#include <tgmath.h>

#define N_MAX_Q1 17 /* up to N = 16 */

#define REAL double
#define SFX _d
#include "oracle_impl.inc"
#undef REAL
#undef SFX

#define REAL long double
#define SFX _ld
#include "oracle_impl.inc"
#undef REAL
#undef SFX

/* size of long double in bytes, so the Python side can marshal it */
int ora_sizeof_long_double(void) { return (int)sizeof(long double); }

int ora_max_threads(void)
{
#if defined(_OPENMP)
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
