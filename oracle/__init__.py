"""CPU oracle of the QSA step.  Test infrastructure only: the library never
imports it; tests, the smoke check and the benchmark's CPU-baseline leg do."""
from .qsa_oracle import *  # noqa: F401,F403
