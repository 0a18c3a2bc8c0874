"""Product quantisation of middle-tier V (oracle).

THIS IS TEST INFRASTRUCTURE (see the package header): only tests, the smoke check and the
benchmark's CPU legs may use it.

FADE-zh §高级功能 / §产品量化 (and FADE-en, its list of advanced features): as an alternative to
INT2, V can be product-quantised at about 2 bits per element; a codebook is trained from
calibration vectors with 256 centroids ("num_centroids=256", "sub_dim=32"), vectors are
encoded to uint8 codes and decoded back to floats.

Readings (the pages give the API and the rate only):
  * one uint8 code (256 centroids) stands for SUB = 4 consecutive channels, so the rate is
    8 / 4 = 2 bits per element, the pages' figure; at head_dim 128 that makes 32 sub-spaces,
    the pages' "32". The other reading (sub-vectors of 32 channels, 0.25 bits per element)
    contradicts the stated rate and is not built;
  * one codebook per layer, shared by every row and KV head: fp16 [d/4][256][4]; the code of
    sub-space s of a vector sits in byte s of its row, so a PQ row has the byte size of an
    INT2 row (d/4 bytes) and carries no scales;
  * encoding picks the centroid at the smallest squared distance. That choice yields an
    integer, so it is taken in one fixed precision on every side: fp32, with
    e_j = x_j - c_j rounded, each square rounded, and the sum taken in channel order
    ((e0^2 + e1^2) + e2^2) + e3^2, each addition rounded; ties go to the lowest index;
  * training is Lloyd's k-means in each sub-space: the centroids start at the sub-vectors of
    the calibration rows ``init_idx`` (the caller's random draw), then each of ``iters``
    rounds assigns every calibration sub-vector by the encoding rule and replaces each
    centroid with the mean of its members: the sum is exact (fp16 values are multiples of
    2^-24 below 2^16, so up to 8192 of them sum exactly in fp64), divided once in fp64 and
    rounded to fp16 (nearest even); a centroid with no member keeps its value;
  * decoded value = the centroid's fp16 channels, exactly.
Pinned by: brute-force nearest search against fp64 distances on separated centroids, tie
order, decode(encode(centroid)) identity, Lloyd rounds on hand-built clusters with known
means, the empty-cluster rule, the rate, and the unit cache's middle values after demotion
equal to decode(encode(v)) of the demoted tokens.
"""

from __future__ import annotations

import numpy as np

SUB = 4              # channels per sub-vector
CENTROIDS = 256      # uint8 codes
MAX_CALIB = 8192     # calibration rows for which the fp64 member sums stay exact


def _split(x16: np.ndarray) -> np.ndarray:
    """fp16 [n, d] -> fp32 [n, d/4, 4] (exact)."""
    x16 = np.asarray(x16, np.float16)
    n, d = x16.shape
    if d % SUB:
        raise ValueError("dim must be a multiple of 4")
    return x16.astype(np.float32).reshape(n, d // SUB, SUB)


def distances(x16: np.ndarray, codebook: np.ndarray) -> np.ndarray:
    """fp32 squared distances [n, d/4, 256] in the fixed order of the encoding rule."""
    xs = _split(x16)                                          # [n, S, 4]
    cb = np.asarray(codebook, np.float16).astype(np.float32)  # [S, 256, 4]
    if cb.shape != (xs.shape[1], CENTROIDS, SUB):
        raise ValueError(f"codebook shape {cb.shape}, expected {(xs.shape[1], CENTROIDS, SUB)}")
    e = (xs[:, :, None, :] - cb[None, :, :, :]).astype(np.float32)   # rounded differences
    sq = (e * e).astype(np.float32)                                  # rounded squares
    acc = sq[..., 0]
    for j in range(1, SUB):                                          # rounded sums, in order
        acc = (acc + sq[..., j]).astype(np.float32)
    return acc


def encode(x16: np.ndarray, codebook: np.ndarray) -> np.ndarray:
    """fp16 [n, d] -> uint8 codes [n, d/4] (nearest centroid, lowest index on ties)."""
    x16 = np.asarray(x16, np.float16)
    out = np.zeros((x16.shape[0], x16.shape[1] // SUB), np.uint8)
    for r in range(0, x16.shape[0], 128):       # rows in blocks, to bound the memory
        out[r:r + 128] = np.argmin(distances(x16[r:r + 128], codebook), axis=-1)  # first min
    return out


def decode(codes: np.ndarray, codebook: np.ndarray) -> np.ndarray:
    """uint8 codes [n, d/4] -> fp16 [n, d] (the centroids' channels)."""
    codes = np.asarray(codes, np.uint8)
    cb = np.asarray(codebook, np.float16)
    n, s = codes.shape
    return cb[np.arange(s)[None, :], codes].reshape(n, s * SUB)


def init_codebook(calib16: np.ndarray, init_idx) -> np.ndarray:
    """Centroid c of every sub-space starts at calibration row init_idx[c]."""
    xs = np.asarray(calib16, np.float16)
    idx = np.asarray(init_idx, np.int64)
    if idx.shape != (CENTROIDS,) or idx.min() < 0 or idx.max() >= xs.shape[0]:
        raise ValueError("init_idx must hold 256 row indices of the calibration set")
    n, d = xs.shape
    return xs[idx].reshape(CENTROIDS, d // SUB, SUB).transpose(1, 0, 2).copy()


def lloyd_round(calib16: np.ndarray, codebook: np.ndarray) -> np.ndarray:
    """One k-means round: assign by the encoding rule, move each centroid to the fp16-rounded
    exact mean of its members; empty centroids stay."""
    xs = _split(calib16).astype(np.float64)          # exact
    codes = encode(calib16, codebook).astype(np.int64)   # [n, S]
    cb = np.asarray(codebook, np.float16).copy()
    n, S = codes.shape
    sub = np.broadcast_to(np.arange(S), (n, S))
    total = np.zeros((S, CENTROIDS, SUB), np.float64)
    count = np.zeros((S, CENTROIDS), np.int64)
    np.add.at(total, (sub, codes), xs)               # exact, so the order is immaterial
    np.add.at(count, (sub, codes), 1)
    hit = count > 0
    cb[hit] = (total[hit] / count[hit][:, None].astype(np.float64)).astype(np.float16)
    return cb


def train(calib16: np.ndarray, init_idx, iters: int) -> np.ndarray:
    """PQ codebook fp16 [d/4][256][4] after ``iters`` Lloyd rounds."""
    calib16 = np.asarray(calib16, np.float16)
    if not 0 < calib16.shape[0] <= MAX_CALIB:
        raise ValueError(f"calibration rows must be in [1, {MAX_CALIB}]")
    cb = init_codebook(calib16, init_idx)
    for _ in range(int(iters)):
        cb = lloyd_round(calib16, cb)
    return cb


def bits_per_element() -> float:
    return 8.0 / SUB
