// Decode step for r = Hq / Hkv = 1 (one translation unit per head ratio, so
// the variants compile in parallel).
#include "hsq_decode.cuh"

HSQ_DEFINE_DECODE(1)
