"""arf: the all-reduce fusion epilogue (kAllReduce, kARResidualRMSNorm) on one GB300."""
