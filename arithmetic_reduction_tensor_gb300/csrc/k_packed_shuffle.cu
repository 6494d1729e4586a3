// k_packed_shuffle.cu -- SHUFFLE_TREE short rows (one-warp team), several
// to a warp group (packed.cuh); the same instances as k_packed_fixed.cu.
#define TCR_PACKED_MODE kPackedShuffle
#define TCR_PACKED_PICK packed_pick_shuffle
#include "k_packed_fixed.cu"
