// bq_multi_q8_0_r1.cu -- Q8_0 instances of the multi-op streaming kernel:
// decode and gate+up (R = 1: row mode, NR = 1, NR = 2, and NR = 3, the paired
// gate+up instance).
#include "bq_multi_launch.cuh"

BQ_MULTI_UNIT(q8_0, bq::QT_Q8_0, r1,
              BQ_INST(bq::QT_Q8_0, 0, 1),
              BQ_INST(bq::QT_Q8_0, 1, 1),
              BQ_INST(bq::QT_Q8_0, 2, 1),
              BQ_INST(bq::QT_Q8_0, 3, 1))
