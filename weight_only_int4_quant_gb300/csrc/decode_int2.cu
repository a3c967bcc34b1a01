// INT2 forms of the decode kernel: the same source as decode.cu, compiled as a
// translation unit of its own so that the INT4 and INT2 kernels build in
// parallel.  launch_decode (decode.cu) calls launch_decode_int2 for INT2.
#define TLQ_DECODE_INT2_UNIT 1
#include "decode.cu"
