// gemm_cfg.h -- build-time shape of the CTA-pair operand pipeline shared by
// the two tensor-core kernels (ag_gemm.cu, gemm_rs.cu).
#pragma once

// K depth of one operand stage (64 or 128 columns; each 64-column block is
// one 128-byte-swizzled sub-tile) and the number of stages in the ring.
// A stage holds, per CTA, its 128 rows of the A block and its 128 rows of
// the B block: (RC_GEMM_PAIR_BK / 64) x 32 KiB.  Measured on GB300
// (8192x4096x4096 bf16): K=128 x 3 stages 0.1729 ms (ag_gemm) / 0.1760 ms
// (gemm_rs); K=64 x 6 stages 0.1861 / 0.1838; K=64 x 5 0.1802 / 0.1852;
// K=64 x 4 0.1918 / 0.1873.
#ifndef RC_GEMM_PAIR_BK
#define RC_GEMM_PAIR_BK 128
#endif
#ifndef RC_GEMM_PAIR_STAGES
#define RC_GEMM_PAIR_STAGES 3
#endif
static_assert(RC_GEMM_PAIR_BK == 64 || RC_GEMM_PAIR_BK == 128, "stage depth is one or two 64-column blocks");
static_assert(RC_GEMM_PAIR_STAGES >= 2 && RC_GEMM_PAIR_STAGES * RC_GEMM_PAIR_BK <= 384,
              "the stage ring must fit in shared memory");
