// Device-side status bits shared by the kernels and the host library.  The
// kernels OR these into a 32-bit word in the caller's workspace; the host maps
// the word to a coda_status with coda_get_status().
#pragma once

#define CODA_DEV_TIMEOUT 0x1         // a bounded mbarrier wait ran out
#define CODA_DEV_LABEL_RANGE 0x2     // a label outside [0, V) that is not ignore_index
#define CODA_DEV_POSITION_RANGE 0x4  // a RoPE position outside [0, max_pos)
