// bq_gemv_q8_0.cu -- Q8_0: generic kernel, stream executor, multi-op dispatch
// and the format's device error word (bq_format_unit.cuh).
#include "bq_format_unit.cuh"

BQ_FORMAT_UNIT(q8_0, bq::QT_Q8_0)
