// bq_multi_q4_k_r234.cu -- Q4_K instances of the multi-op streaming kernel:
// verify with R = 2, 3, 4 (one weight row per lane).
#include "bq_multi_launch.cuh"

BQ_MULTI_UNIT(q4_k, bq::QT_Q4_K, r234,
              BQ_INST(bq::QT_Q4_K, 1, 2),
              BQ_INST(bq::QT_Q4_K, 1, 3),
              BQ_INST(bq::QT_Q4_K, 1, 4))
