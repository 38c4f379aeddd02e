// Device status bits recorded in the first word of every workspace.
#pragma once

#define FA_STATUS_TIMEOUT_LOAD 0x1      // a load (TMA producer) wait ran out
#define FA_STATUS_TIMEOUT_MMA 0x2       // the MMA issuer's wait ran out
#define FA_STATUS_TIMEOUT_SOFTMAX 0x4   // a softmax / gradient warp's wait ran out
#define FA_STATUS_TIMEOUT_UNIT 0x8      // the work-unit hand-off wait ran out
#define FA_STATUS_TIMEOUT_DRAIN 0x10    // copies in flight did not land before exit
#define FA_STATUS_TIMEOUT_MASK 0xff
#define FA_STATUS_BAD_INPUT 0x100       // paged decode: a length outside [1, Nk] or a page index out of range

// Workspace header: [0] status word, [4] spare, [8..] per-kernel unit counters.
#define FA_WS_STATUS_OFFSET 0
#define FA_WS_COUNTER_OFFSET 16
#define FA_WS_HEADER_BYTES 256
