// profile.h -- launch bracketing for dspark_profile_* (host side).
#pragma once
#include <cuda_runtime.h>

namespace dspark {

enum ProfName : int {
    kPDraftPrep = 0,
    kPDraftSweepGeneric = 1,
    kPDraftSweepTc = 2,
    kPVerifyPass1 = 3,
    kPVerifyAccept = 4,
    kPVerifyResidualGeneric = 5,
    kPVerifyResidualTc = 6,
    kPVerifySample = 7,
    kPSchedule = 8,
    kPDraftPrepRnn = 9,
    kPDraftRnnGru = 10,
    kPScheduleThreshold = 11,
    kPStsHist = 12,
    kPStsEce = 13,
    kPStsAdvance = 14,
    kPStsApply = 15,
    kPStsFix = 16,
    kPDraftRnnGruFinish = 17,
};

void prof_begin(int name, cudaStream_t s);
void prof_end(cudaStream_t s);

}  // namespace dspark
