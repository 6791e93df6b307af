// bq_multi_q4_0_r234.cu -- Q4_0 instances of the multi-op streaming kernel:
// verify with R = 2, 3, 4 (NR = 1, 2).
#include "bq_multi_launch.cuh"

BQ_MULTI_UNIT(q4_0, bq::QT_Q4_0, r234,
              BQ_INST(bq::QT_Q4_0, 1, 2),
              BQ_INST(bq::QT_Q4_0, 2, 2),
              BQ_INST(bq::QT_Q4_0, 1, 3),
              BQ_INST(bq::QT_Q4_0, 2, 3),
              BQ_INST(bq::QT_Q4_0, 1, 4),
              BQ_INST(bq::QT_Q4_0, 2, 4))
