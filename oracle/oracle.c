/*
 * Oracle for the five-point Jacobi solver of implicit 2-D diffusion.
 *
 * TEST INFRASTRUCTURE ONLY: a plain, slow, single-threaded CPU restatement
 * of what the method computes, used by tests/, the smoke check and the
 * CPU-baseline leg of the benchmark. The CUDA library does not include, link
 * or call anything here, and this file shares no code with it.
 *
 * Source: "Synchronous vs block-async Jacobi on one RTX 5050"
 * (stencil-jacobian.vercel.app), sections 01 "The problem" and 02 "Method".
 *
 * Build: cc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared
 * -pthread (no multiply-add contraction, IEEE subnormals kept; see
 * oracle/__init__.py). The single-threaded functions are the oracle of
 * record; the *_mt forms split a sweep's rows among POSIX threads and give
 * the same bits (checked in tests/test_oracle_threads.py).
 *
 * Parity status of each function is recorded in oracle/__init__.py's header.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#if defined(__FAST_MATH__)
#error "the oracle must not be built with fast-math"
#endif

#define REAL float
#define SFX f32
#include "oracle_body.h"
#undef REAL
#undef SFX

#define REAL double
#define SFX f64
#include "oracle_body.h"
#undef REAL
#undef SFX
