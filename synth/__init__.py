"""Seeded synthetic inputs (weights, token ids, test vectors) shared by the
oracle side and the CUDA side.  Holds no arithmetic of the decode step."""
