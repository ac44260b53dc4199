"""CPU oracle of the KV-cache codec -- test infrastructure only (see
``oracle.py``)."""
