// Built launch plans: X(id, V, S, P, K, C).
//
//   V  elements per vector access (4 = float4 body with scalar head/tail,
//      1 = scalar, for pointers whose 16-byte phases differ)
//   S  warps per program (W = 32*S cooperating workers per row)
//   P  programs (rows) packed per CTA, T = 32*S*P threads
//   K  V-vectors per worker: the register stripe holds K*V floats
//   C  CTAs per row (a thread-block cluster when C > 1)
//
// A plan covers a row of `width` when its workers can own every element:
// V = 4: floor(width/4) <= K*W*C (head/tail scalars are extra);
// V = 1: width <= K*W*C.
//
// The selector in tile_api.cu picks from this table by width and row count;
// every plan can also be forced through tile_run_plan_f32 (plan sweeps and
// the per-plan parity tests use that).
#pragma once

#define TILE_PLAN_LIST(X)                                                     \
    /* one warp per row, packed 4-8 rows per CTA */                           \
    X(0, 4, 1, 8, 1, 1)                                                       \
    X(1, 4, 1, 8, 2, 1)                                                       \
    X(2, 4, 1, 4, 4, 1)                                                       \
    /* 2-8 warps per row, packed */                                           \
    X(3, 4, 2, 4, 4, 1)                                                       \
    X(4, 4, 2, 2, 4, 1)                                                       \
    X(5, 4, 4, 2, 4, 1)                                                       \
    X(6, 4, 4, 1, 4, 1)                                                       \
    X(7, 4, 4, 1, 8, 1)                                                       \
    X(8, 4, 8, 1, 4, 1)                                                       \
    X(9, 4, 16, 1, 2, 1)                                                      \
    X(10, 4, 8, 1, 8, 1)                                                      \
    X(11, 4, 16, 1, 4, 1)                                                     \
    X(12, 4, 32, 1, 2, 1)                                                     \
    X(13, 4, 32, 1, 4, 1)                                                     \
    X(14, 4, 16, 1, 8, 1)                                                     \
    /* one row over a cluster of 2-8 CTAs */                                  \
    X(15, 4, 16, 1, 4, 2)                                                     \
    X(16, 4, 16, 1, 4, 4)                                                     \
    X(17, 4, 8, 1, 8, 4)                                                      \
    X(18, 4, 16, 1, 4, 8)                                                     \
    X(19, 4, 8, 1, 8, 8)                                                      \
    X(20, 4, 32, 1, 4, 8)                                                     \
    /* more packings around the common widths */                              \
    X(21, 4, 4, 4, 2, 1)                                                      \
    X(22, 4, 8, 2, 2, 1)                                                      \
    X(23, 4, 32, 1, 1, 1)                                                     \
    X(24, 4, 8, 2, 4, 1)                                                      \
    /* scalar plans for pointers that are not co-aligned */                   \
    X(25, 1, 1, 8, 4, 1)                                                      \
    X(26, 1, 4, 2, 8, 1)                                                      \
    X(27, 1, 8, 1, 16, 1)                                                     \
    X(28, 1, 32, 1, 16, 1)                                                    \
    X(29, 1, 32, 1, 16, 8)                                                    \
    /* deeper stripes: more loads in flight per thread */                     \
    X(30, 4, 16, 1, 8, 8)                                                     \
    X(31, 4, 8, 1, 16, 1)                                                     \
    X(32, 4, 4, 1, 16, 1)                                                     \
    X(33, 4, 16, 1, 8, 4)                                                     \
    X(34, 4, 16, 1, 8, 2)                                                     \
    X(35, 4, 2, 1, 16, 1)                                                     \
    X(36, 4, 4, 2, 8, 1)                                                      \
    /* fewer workers, deeper stripes (packed BF16 rows of 2048-4096) */       \
    X(37, 4, 2, 1, 8, 1)                                                      \
    X(38, 4, 2, 2, 8, 1)                                                      \
    X(39, 4, 1, 4, 8, 1)

#define TILE_PLAN_COUNT 40

// Shared-memory-staged plans (staged_kernel.cuh): X(id, S, K, KB), one row
// per CTA iteration (P = 1, C = 1), 16-byte vectors, persistent grid; KB is
// the shared memory a CTA gives to its ring of stages (between 1 and 8 rows,
// so a smaller budget means more CTAs, and warps, per SM).  Their ids follow
// the register plans.
#define TILE_STAGED_LIST(X) \
    X(40, 4, 4, 100)        \
    X(41, 4, 8, 100)        \
    X(42, 8, 4, 100)        \
    X(43, 8, 8, 100)        \
    X(44, 4, 4, 48)         \
    X(45, 4, 8, 48)         \
    X(46, 2, 8, 32)         \
    X(47, 4, 4, 32)         \
    /* more workers, shorter stripes: fewer gamma/beta registers per    */ \
    /* thread where the 2-byte affine rows keep them across rows        */ \
    X(48, 8, 2, 48)         \
    X(49, 8, 2, 96)         \
    X(50, 16, 1, 64)        \
    X(51, 16, 2, 100)       \
    X(52, 4, 2, 32)

#define TILE_STAGED_COUNT 13

// R-rows-per-CTA plans (multi_kernel.cuh): X(id, S, K, R), a CTA of 32*S
// threads normalising R rows, every thread owning the same columns of each
// (K 16-byte vectors per row), so reductions and gamma/beta loads serve R
// rows.  16-byte vectors on aligned rows of whole vectors, as the staged
// plans; their ids follow the staged plans.
#define TILE_MULTI_LIST(X) \
    X(53, 4, 4, 2)         \
    X(54, 8, 2, 2)         \
    X(55, 8, 4, 2)         \
    X(56, 16, 1, 2)        \
    X(57, 8, 2, 4)         \
    X(58, 16, 2, 2)        \
    X(59, 4, 2, 4)         \
    X(60, 16, 4, 2)

#define TILE_MULTI_COUNT 8

// Widest row covered by both a V = 4 and a V = 1 plan.
#define TILE_MAX_WIDTH 131072
