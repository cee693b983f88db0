"""Random rotations (oracle, fp64).

Test infrastructure only (see ``oracle/__init__.py``).

Sources
-------
* Haar rotation: QR decomposition of a d×d i.i.d. Gaussian matrix, keeping the
  orthogonal factor; generated once from a fixed seed and shared by every
  vector: "TurboQuant 详解", section "TurboQuant_mse 的官方步骤" (step 1);
  "turboquant-first-principles-walkthrough", section "核心洞察" and
  "部署参数与系统集成要点" (fixed seed).
* Randomized Walsh-Hadamard rotation as the structured alternative:
  "TurboQuant 和 RotorQuant 的真相", chapter 3 (WHT, O(d log d)) and
  chapter 7 ("WHT vs Random Rotation").

Readings where the pages are silent or ambiguous:
* The QR factor is sign-fixed, Π = Q · diag(sign(diag R)) with sign(0) = +1,
  which makes Π Haar-distributed and makes ΠᵀG upper triangular with a
  positive diagonal.
* Hadamard orders that are not powers of two (1536 = 12·128, 3072 = 12·256)
  use H_12 ⊗ H_{2^k}, H_12 the Paley matrix built from the quadratic residues
  modulo 11 and H_{2^k} the Sylvester matrix; the randomized rotation is
  Π = (1/√d) · H · diag(σ), σ_i = ±1.
"""

import math

import numpy as np


def haar_rotation(G):
    """Π = Q · diag(sign(diag R)) for the QR decomposition G = QR."""
    G = np.asarray(G, dtype=np.float64)
    Q, R = np.linalg.qr(G)
    sgn = np.where(np.diag(R) < 0.0, -1.0, 1.0)
    return Q * sgn[None, :]


def sylvester_hadamard(n):
    """H_n for n a power of two, H_{2m} = [[H_m, H_m], [H_m, -H_m]]."""
    if n < 1 or (n & (n - 1)) != 0:
        raise ValueError("n must be a power of two")
    H = np.ones((1, 1), dtype=np.float64)
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H


def paley_hadamard_12():
    """Paley construction I for q = 11: H = I + [[0, 1ᵀ], [-1, Q]].

    Q is the Jacobsthal matrix Q_ij = χ(j - i), χ the quadratic character
    modulo 11 (χ(0) = 0).  q ≡ 3 (mod 4) makes the bordered matrix
    skew-symmetric, so H Hᵀ = 12 I.
    """
    q = 11
    residues = {(x * x) % q for x in range(1, q)}
    chi = np.array([0.0] + [1.0 if a in residues else -1.0 for a in range(1, q)])
    Q = np.empty((q, q), dtype=np.float64)
    for i in range(q):
        for j in range(q):
            Q[i, j] = chi[(j - i) % q]
    S = np.zeros((q + 1, q + 1), dtype=np.float64)
    S[0, 1:] = 1.0
    S[1:, 0] = -1.0
    S[1:, 1:] = Q
    return np.eye(q + 1) + S


def hadamard(d):
    """Hadamard matrix of order d = 2^k, or d = 12 · 2^k as H_12 ⊗ H_{2^k}.

    Index convention of the Kronecker product: row i = 2^k · a + j with
    a the H_12 index and j the Sylvester index.
    """
    if d >= 1 and (d & (d - 1)) == 0:
        return sylvester_hadamard(d)
    if d % 12 == 0:
        m = d // 12
        if m >= 1 and (m & (m - 1)) == 0:
            return np.kron(paley_hadamard_12(), sylvester_hadamard(m))
    raise ValueError("Hadamard order must be 2^k or 12*2^k")


def hadamard_rotation(d, signs):
    """Randomized Hadamard rotation Π = (1/√d) · H · diag(σ)."""
    signs = np.asarray(signs, dtype=np.float64)
    return hadamard(d) * signs[None, :] / math.sqrt(d)
